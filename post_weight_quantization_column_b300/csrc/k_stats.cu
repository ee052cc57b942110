// Step 1: per-input-channel statistic a_j = (1/N) sum_r |X[r, j]|.
// "AWQ (Activation-aware Weight Quantization)", 技术原理 - 重要通道识别的统计依据;
// aiqz.cc article "awq-activation-aware-quantization", section 1 (I_i = E|X_i|).
//
// HBM-bound column reduction.  A CTA owns 256 consecutive channels and one
// slice of rows.  Its producer thread streams the slice through a 6-stage
// ring of 32-row x 256-channel boxes (one 16 KB tensor copy each), so a CTA
// keeps 96 KB of X in flight with one instruction per box and the loads do
// not depend on the SM's issue rate; two CTAs share an SM.  Eight consumer warps take interleaved
// rows of each box: lane l adds the 8 channels 8l .. 8l+7.  Rows past N and
// channels past D arrive as zeros.  Per-thread sums are fp32, the 8 warps are combined in
// a fixed order through shared memory, and the row slices are summed in a
// fixed fp32 tree by the last CTA of each column chunk to finish (a per-chunk
// ticket counter), so the result does not depend on timing.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {

namespace {

constexpr int kBoxBytes = kStatsBoxRows * kStatsCols * 2;  // 16 KB
constexpr int kStatsSmem = kStatsStages * kBoxBytes;

// |lo| and |hi| of a packed bf16 pair, widened exactly to fp32.
__device__ __forceinline__ void add_abs_pair(uint32_t u, float& a0, float& a1) {
  a0 += __uint_as_float((u << 16) & 0x7FFFFFFFu);
  a1 += __uint_as_float(u & 0x7FFF0000u);
}

__device__ __forceinline__ void add_abs_vec(const uint4& v, float (&acc)[8]) {
  add_abs_pair(v.x, acc[0], acc[1]);
  add_abs_pair(v.y, acc[2], acc[3]);
  add_abs_pair(v.z, acc[4], acc[5]);
  add_abs_pair(v.w, acc[6], acc[7]);
}

// The same, also keeping the running max of |x| per channel (exact).
__device__ __forceinline__ void add_max_abs_pair(uint32_t u, float& a0, float& a1, float& m0, float& m1) {
  const float x0 = __uint_as_float((u << 16) & 0x7FFFFFFFu);
  const float x1 = __uint_as_float(u & 0x7FFF0000u);
  a0 += x0;
  a1 += x1;
  m0 = fmaxf(m0, x0);
  m1 = fmaxf(m1, x1);
}

template <bool kMax>
__device__ __forceinline__ void add_vec(const uint4& v, float (&acc)[8], float (&mx)[8]) {
  if (kMax) {
    add_max_abs_pair(v.x, acc[0], acc[1], mx[0], mx[1]);
    add_max_abs_pair(v.y, acc[2], acc[3], mx[2], mx[3]);
    add_max_abs_pair(v.z, acc[4], acc[5], mx[4], mx[5]);
    add_max_abs_pair(v.w, acc[6], acc[7], mx[6], mx[7]);
  } else {
    add_abs_vec(v, acc);
  }
}

}  // namespace

// mean_abs: written with the mean when sum_abs is null.  sum_abs: when given,
// the slice total of each channel (float64) is added to it instead.  max_abs:
// when kMax, max(max_abs, the batch's max |x|) is stored back.  nan_on_error:
// the last CTA of a chunk writes NaN means when the status word is set (a row
// slice of the chunk gave up a wait and its partial sums are incomplete), for
// callers that have no status word of their own to read.
template <bool kMax>
__global__ void __launch_bounds__(kStatsThreads) act_stats_kernel(const __grid_constant__ CUtensorMap tmX, int64_t N,
                                                                 int64_t D, int64_t rows_per_split,
                                                                 float* __restrict__ partial,
                                                                 float* __restrict__ partial_max,
                                                                 unsigned int* __restrict__ tickets,
                                                                 float* __restrict__ mean_abs,
                                                                 double* __restrict__ sum_abs,
                                                                 float* __restrict__ max_abs, uint32_t* status,
                                                                 int nan_on_error) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) float red[kStatsRowLanes][kStatsCols];
  __shared__ __align__(8) uint64_t full_bar[kStatsStages];
  __shared__ __align__(8) uint64_t empty_bar[kStatsStages];
  __shared__ int abort_sh;
  __shared__ bool last;
  volatile int* abort_flag = &abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kStatsCols;
  const int width = static_cast<int>(min(static_cast<int64_t>(kStatsCols), D - c0));  // channels of this chunk
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_split;
  const int64_t r1 = min(N, r0 + rows_per_split);
  const int nbox = static_cast<int>((r1 - r0 + kStatsBoxRows - 1) / kStatsBoxRows);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStatsStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kStatsRowLanes);
    }
    abort_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();

  float acc[8], mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = mx[i] = 0.f;

  if (warp == kStatsRowLanes) {
    // ------------------------------------------------------------ producer
    // rows_per_split is a multiple of the box height, so a box never reaches
    // into the next slice; the last slice's boxes end in zero fill past N
    if (lane == 0) {
      prefetch_tmap(&tmX);
      int b = 0;
      for (; b < nbox; ++b) {
        const int s = b % kStatsStages;
        if (b >= kStatsStages && !mbar_wait(&empty_bar[s], ((b / kStatsStages) + 1) & 1, status, abort_flag)) break;
        mbar_arrive_expect_tx(&full_bar[s], kBoxBytes);
        tma_load_2d(ring + s * kBoxBytes, &tmX, &full_bar[s], static_cast<int32_t>(c0),
                    static_cast<int32_t>(r0 + static_cast<int64_t>(b) * kStatsBoxRows));
      }
      // after an abort, the copies still in flight into this CTA land before
      // it moves on (boxes b - kStatsStages .. b - 1 may not have been consumed)
      if (b < nbox || *abort_flag)
        for (int j = max(0, b - kStatsStages); j < b; ++j)
          mbar_wait(&full_bar[j % kStatsStages], (j / kStatsStages) & 1, nullptr, nullptr);
    }
  } else {
    // ------------------------------------------------------------ consumer warps
    const bool active = lane * 8 < width;
    for (int b = 0; b < nbox; ++b) {
      const int s = b % kStatsStages;
      if (!mbar_wait(&full_bar[s], (b / kStatsStages) & 1, status, abort_flag)) break;
      const int64_t rb = r0 + static_cast<int64_t>(b) * kStatsBoxRows;
      const int rows = static_cast<int>(min(static_cast<int64_t>(kStatsBoxRows), r1 - rb));
      const uint8_t* st = ring + s * kBoxBytes + lane * 16;
      if (active) {
        if (rows == kStatsBoxRows) {
          uint4 v[kStatsBoxRows / kStatsRowLanes];
#pragma unroll
          for (int i = 0; i < kStatsBoxRows / kStatsRowLanes; ++i)
            v[i] = *reinterpret_cast<const uint4*>(st + (warp + i * kStatsRowLanes) * (kStatsCols * 2));
#pragma unroll
          for (int i = 0; i < kStatsBoxRows / kStatsRowLanes; ++i) add_vec<kMax>(v[i], acc, mx);
        } else {
          for (int r = warp; r < rows; r += kStatsRowLanes)
            add_vec<kMax>(*reinterpret_cast<const uint4*>(st + r * (kStatsCols * 2)), acc, mx);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
  }

  if (warp < kStatsRowLanes) {
    float4* dst = reinterpret_cast<float4*>(&red[warp][lane * 8]);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  __syncthreads();
  const int t = threadIdx.x;
  const int64_t j = c0 + t;
  if (t < kStatsCols && t < width) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kStatsRowLanes; ++k) sum += red[k][t];
    partial[static_cast<int64_t>(blockIdx.y) * D + j] = sum;
  }
  if (kMax) {
    __syncthreads();
    if (warp < kStatsRowLanes) {
      float4* dst = reinterpret_cast<float4*>(&red[warp][lane * 8]);
      dst[0] = make_float4(mx[0], mx[1], mx[2], mx[3]);
      dst[1] = make_float4(mx[4], mx[5], mx[6], mx[7]);
    }
    __syncthreads();
    if (t < kStatsCols && t < width) {
      float m = 0.f;
#pragma unroll
      for (int k = 0; k < kStatsRowLanes; ++k) m = fmaxf(m, red[k][t]);
      partial_max[static_cast<int64_t>(blockIdx.y) * D + j] = m;
    }
  }
  // the last row slice of this column chunk to finish sums the slices
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&tickets[blockIdx.x], 1u) == gridDim.y - 1u;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // a slice that timed out set the status word before its ticket
  const bool poison = nan_on_error && status && *reinterpret_cast<volatile uint32_t*>(status) != 0u;
  if (t < kStatsCols && t < width) {
    // the slices in batches of 32 (one batch unless the grid has more than
    // 32 slices), each batch as a fixed pairwise tree in fp32, the batches in
    // order: the error stays below (5 + batches) * 2^-24 of the total, and
    // no fp64 arithmetic (slow on this part) sits on the kernel's tail
    const int splits = static_cast<int>(gridDim.y);
    float s = 0.f;
    for (int k = 0; k < splits; k += 32) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = k + i < splits ? partial[static_cast<int64_t>(k + i) * D + j] : 0.f;
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) v[i] += v[i + w];
      s += v[0];
    }
    if (!isfinite(s)) set_error(status, AWQ_DEV_NONFINITE);
    if (sum_abs) {
      sum_abs[j] += static_cast<double>(s);  // this CTA alone owns channel j now
    } else {
      mean_abs[j] = poison ? __int_as_float(0x7FC00000) : __fdiv_rn(s, static_cast<float>(N));
    }
    if (kMax) {
      float m = max_abs[j];
      for (int k = 0; k < splits; ++k) m = fmaxf(m, partial_max[static_cast<int64_t>(k) * D + j]);
      max_abs[j] = m;
    }
  }
  if (t == 0) tickets[blockIdx.x] = 0u;  // ready for the next call
}

// mean = fp32(total / rows) after a stream of accumulated batches.
__global__ void stats_finalize_kernel(const double* __restrict__ sum_abs, int64_t rows, int64_t D,
                                      float* __restrict__ mean_abs) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j < D) mean_abs[j] = static_cast<float>(sum_abs[j] / static_cast<double>(rows));
}

void stats_plan(int64_t N, int64_t D, int* splits, int64_t* rows_per_split) {
  const int64_t chunks = (D + kStatsCols - 1) / kStatsCols;
  // as many row slices as keep the grid within one resident wave
  int64_t want = kStatsTargetCtas / (chunks > 0 ? chunks : 1);
  const int64_t max_splits = (N + 4 * kStatsBoxRows - 1) / (4 * kStatsBoxRows);  // >= 4 boxes per slice
  if (want > max_splits) want = max_splits;
  if (want < 1) want = 1;
  if (want > kStatsMaxSplits) want = kStatsMaxSplits;
  int64_t rps = (N + want - 1) / want;
  rps = (rps + kStatsBoxRows - 1) / kStatsBoxRows * kStatsBoxRows;
  *rows_per_split = rps;
  *splits = static_cast<int>((N + rps - 1) / rps);
  if (*splits < 1) *splits = 1;
}

cudaError_t launch_act_stats(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, int64_t N, int64_t D,
                             int64_t ldx, float* mean_abs, double* sum_abs, float* max_abs, float* partial,
                             float* partial_max, unsigned int* tickets, int splits, int64_t rows_per_split,
                             uint32_t* status, int nan_on_error, cudaStream_t stream) {
  CUtensorMap tm;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
  const cuuint32_t box[2] = {kStatsCols, kStatsBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(stats_chunks(D)), static_cast<unsigned>(splits));
  if (max_abs) {
    cudaError_t e = cudaFuncSetAttribute(act_stats_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kStatsSmem);
    if (e != cudaSuccess) return e;
    act_stats_kernel<true><<<grid, kStatsThreads, kStatsSmem, stream>>>(
        tm, N, D, rows_per_split, partial, partial_max, tickets, mean_abs, sum_abs, max_abs, status, nan_on_error);
  } else {
    cudaError_t e = cudaFuncSetAttribute(act_stats_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kStatsSmem);
    if (e != cudaSuccess) return e;
    act_stats_kernel<false><<<grid, kStatsThreads, kStatsSmem, stream>>>(
        tm, N, D, rows_per_split, partial, partial_max, tickets, mean_abs, sum_abs, max_abs, status, nan_on_error);
  }
  return cudaGetLastError();
}

cudaError_t launch_stats_finalize(const double* sum_abs, int64_t rows, int64_t D, float* mean_abs,
                                  cudaStream_t stream) {
  stats_finalize_kernel<<<static_cast<unsigned>((D + 255) / 256), 256, 0, stream>>>(sum_abs, rows, D, mean_abs);
  return cudaGetLastError();
}

int64_t stats_chunks(int64_t D) { return (D + kStatsCols - 1) / kStatsCols; }

}  // namespace awqdev
