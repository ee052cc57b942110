// Step 1: per-input-channel statistic a_j = (1/N) sum_r |X[r, j]|.
// "AWQ (Activation-aware Weight Quantization)", 技术原理 - 重要通道识别的统计依据;
// aiqz.cc article "awq-activation-aware-quantization", section 1 (I_i = E|X_i|).
//
// HBM-bound column reduction.  A CTA owns 256 consecutive channels: each lane
// of a warp reads one 16-byte vector (8 bf16 channels) of a row, so a warp
// reads 512 contiguous bytes per row; the 8 warps take interleaved rows of the
// CTA's row slice.  Per-thread sums are fp32, the 8 warps are combined in a
// fixed order through shared memory, and the row slices are summed in fp64 in
// slice order by the last CTA of each column chunk to finish (a per-chunk
// ticket counter), so the result does not depend on timing.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

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

__global__ void __launch_bounds__(kStatsThreads) act_stats_kernel(const __nv_bfloat16* __restrict__ X, int64_t N,
                                                                 int64_t D, int64_t ldx, int64_t rows_per_split,
                                                                 float* __restrict__ partial,
                                                                 unsigned int* __restrict__ tickets,
                                                                 float* __restrict__ mean_abs, uint32_t* status) {
  __shared__ __align__(16) float red[kStatsRowLanes][kStatsCols];
  __shared__ bool last;
  const int lane = threadIdx.x & 31;
  const int rl = threadIdx.x >> 5;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * kStatsCols + lane * 8;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_split;
  const int64_t r1 = min(N, r0 + rows_per_split);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (col < D) {
    const __nv_bfloat16* base = X + col;
    int64_t r = r0 + rl;
    constexpr int S = kStatsRowLanes;
    // 8 rows in flight per thread
    for (; r + 7 * S < r1; r += 8 * S) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ld_stream_v4(base + (r + i * S) * ldx);
#pragma unroll
      for (int i = 0; i < 8; ++i) add_abs_vec(v[i], acc);
    }
    for (; r < r1; r += S) add_abs_vec(ld_stream_v4(base + r * ldx), acc);
  }
  float4* dst = reinterpret_cast<float4*>(&red[rl][lane * 8]);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  const int t = threadIdx.x;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kStatsCols + t;
  if (t < kStatsCols && j < D) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kStatsRowLanes; ++k) sum += red[k][t];
    partial[static_cast<int64_t>(blockIdx.y) * D + j] = sum;
  }
  // the last row slice of this column chunk to finish sums the slices
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&tickets[blockIdx.x], 1u) == gridDim.y - 1u;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (t < kStatsCols && j < D) {
    const int splits = static_cast<int>(gridDim.y);
    double s = 0.0;
    int k = 0;
    for (; k + 8 <= splits; k += 8) {
      float v[8];  // eight loads in flight, added in slice order
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = partial[static_cast<int64_t>(k + i) * D + j];
#pragma unroll
      for (int i = 0; i < 8; ++i) s += static_cast<double>(v[i]);
    }
    for (; k < splits; ++k) s += static_cast<double>(partial[static_cast<int64_t>(k) * D + j]);
    const float m = static_cast<float>(s / static_cast<double>(N));
    if (!isfinite(m)) set_error(status, AWQ_DEV_NONFINITE);
    mean_abs[j] = m;
  }
  if (t == 0) tickets[blockIdx.x] = 0u;  // ready for the next call
}

void stats_plan(int64_t N, int64_t D, int* splits, int64_t* rows_per_split) {
  const int64_t chunks = (D + kStatsCols - 1) / kStatsCols;
  int64_t want = (kStatsTargetCtas + chunks - 1) / (chunks > 0 ? chunks : 1);
  const int64_t max_splits = (N + 63) / 64;  // at least 64 rows per slice
  if (want > max_splits) want = max_splits;
  if (want < 1) want = 1;
  if (want > kStatsMaxSplits) want = kStatsMaxSplits;
  int64_t rps = (N + want - 1) / want;
  rps = (rps + kStatsRowLanes - 1) / kStatsRowLanes * kStatsRowLanes;
  if (rps < kStatsRowLanes) rps = kStatsRowLanes;
  *rows_per_split = rps;
  *splits = static_cast<int>((N + rps - 1) / rps);
  if (*splits < 1) *splits = 1;
}

cudaError_t launch_act_stats(const void* X, int64_t N, int64_t D, int64_t ldx, float* mean_abs, float* partial,
                             unsigned int* tickets, int splits, int64_t rows_per_split, uint32_t* status,
                             cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(stats_chunks(D)), static_cast<unsigned>(splits));
  act_stats_kernel<<<grid, kStatsThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(X), N, D, ldx, rows_per_split,
                                                       partial, tickets, mean_abs, status);
  return cudaGetLastError();
}

int64_t stats_chunks(int64_t D) { return (D + kStatsCols - 1) / kStatsCols; }

}  // namespace awqdev
