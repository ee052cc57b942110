// Loss reduction and argmin ("AWQ (Activation-aware Weight Quantization)",
// 缩放因子优化的完整流程 steps 4c-6): the search leaves one fp32 sum of squares
// per (candidate, row tile, column); these are summed in a fixed order, first
// over row tiles (per-column losses), then over columns (L_k, fp64), then
// k* = first argmin and s* = s_k* is copied out.
#include "internal.h"
#include "ptx.cuh"

namespace awqdev {

constexpr int kRedThreads = 256;  // threads of the single-CTA selection
constexpr int kRedBlockCols = 256;
constexpr int kRedColsPerThread = 4;
constexpr int kRedSumThreads = kRedBlockCols / kRedColsPerThread;  // 64

// One kernel for the whole reduction.  CTA (bx, k) owns columns
// [256 bx, 256 bx + 256) of candidate k; each of its 64 threads takes 4
// adjacent columns with 16-byte loads (8 loads in flight per run) and sums
// each column over the row tiles into col[k][n] -- each run of 8 tiles as a
// fixed fp32 pairwise tree (error below 3 * 2^-24 of the run's sum of
// squares), the runs in tile order in fp64, which keeps fp64 adds (slow on
// this part) to one per 8 tiles; the CTA then sums its 256 columns in a
// fixed fp64 tree into blk[k][bx].  The last CTA to finish (a ticket
// counter that the caller zeroed) adds blk[k][0..nb) in block order into
// L_k, picks k* = first argmin and copies s* = s_k*.  Every sum has a fixed
// order, so the result does not depend on timing.
__global__ void __launch_bounds__(kRedSumThreads)
    reduce_losses_kernel(const float* __restrict__ partial, int m_tiles, int64_t D_out, int G,
                         double* __restrict__ col, double* __restrict__ blk, unsigned int* __restrict__ ticket,
                         double* __restrict__ losses, int32_t* __restrict__ best_idx, const float* __restrict__ s_tab,
                         int64_t D_in, float* __restrict__ s_star, uint32_t* status) {
  __shared__ double sh[kRedBlockCols];
  __shared__ bool last;
  __shared__ int kbest;
  const int k = blockIdx.y;
  const int nb = gridDim.x;
  const int t = threadIdx.x;
  // D_out is a multiple of 8, so a thread's 4 columns are all inside or all outside
  const int64_t n = static_cast<int64_t>(blockIdx.x) * kRedBlockCols + kRedColsPerThread * t;
  double v[kRedColsPerThread] = {0.0, 0.0, 0.0, 0.0};
  if (n < D_out) {
    const float* p = partial + static_cast<int64_t>(k) * m_tiles * D_out + n;
    for (int m = 0; m < m_tiles; m += 8) {
      float4 x[8];  // eight 16-byte loads in flight; tiles past the end count as 0
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[i] = m + i < m_tiles ? *reinterpret_cast<const float4*>(p + static_cast<int64_t>(m + i) * D_out)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 t4 = make_float4(((x[0].x + x[1].x) + (x[2].x + x[3].x)) + ((x[4].x + x[5].x) + (x[6].x + x[7].x)),
                                    ((x[0].y + x[1].y) + (x[2].y + x[3].y)) + ((x[4].y + x[5].y) + (x[6].y + x[7].y)),
                                    ((x[0].z + x[1].z) + (x[2].z + x[3].z)) + ((x[4].z + x[5].z) + (x[6].z + x[7].z)),
                                    ((x[0].w + x[1].w) + (x[2].w + x[3].w)) + ((x[4].w + x[5].w) + (x[6].w + x[7].w)));
      v[0] += static_cast<double>(t4.x);
      v[1] += static_cast<double>(t4.y);
      v[2] += static_cast<double>(t4.z);
      v[3] += static_cast<double>(t4.w);
    }
    double* cp = col + static_cast<int64_t>(k) * D_out + n;  // caller memory: 8-byte aligned only
#pragma unroll
    for (int c = 0; c < kRedColsPerThread; ++c) cp[c] = v[c];
  }
#pragma unroll
  for (int c = 0; c < kRedColsPerThread; ++c) sh[kRedColsPerThread * t + c] = v[c];
  __syncthreads();
  for (int w = kRedBlockCols / 2; w > 0; w >>= 1) {
    for (int i = t; i < w; i += kRedSumThreads) sh[i] += sh[i + w];
    __syncthreads();
  }
  if (t == 0) {
    blk[static_cast<int64_t>(k) * nb + blockIdx.x] = sh[0];
    __threadfence();
    const unsigned int done = atomicAdd(ticket, 1u);
    last = done == static_cast<unsigned int>(nb) * static_cast<unsigned int>(G) - 1u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (t < G) {  // G <= kMaxGrid = kRedSumThreads
    double L = 0.0;
#pragma unroll 4
    for (int b = 0; b < nb; ++b) L += blk[static_cast<int64_t>(t) * nb + b];
    sh[t] = L;
    losses[t] = L;
  }
  __syncthreads();
  if (t == 0) {
    int b = -1;
    double bl = 0.0;
    for (int kk = 0; kk < G; ++kk) {
      const double L = sh[kk];
      if (isnan(L)) continue;
      if (b < 0 || L < bl) {
        b = kk;
        bl = L;
      }
    }
    if (b < 0) {
      b = 0;
      set_error(status, AWQ_DEV_NONFINITE);
    }
    kbest = b;
    *best_idx = b;
    *ticket = 0u;  // ready for the next call on this workspace
  }
  __syncthreads();
  const float* src = s_tab + static_cast<int64_t>(kbest) * D_in;
  if ((reinterpret_cast<uintptr_t>(s_star) & 15u) == 0 && (D_in & 3) == 0) {
    // s_tab rows start 16-byte aligned (D_in is a multiple of the group size)
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* d4 = reinterpret_cast<float4*>(s_star);
#pragma unroll 4
    for (int64_t j = t; j < D_in / 4; j += kRedSumThreads) d4[j] = s4[j];
  } else {
    for (int64_t j = t; j < D_in; j += kRedSumThreads) s_star[j] = src[j];
  }
}

// The final step of the reduction over block partials gathered from several
// searches of disjoint column slices (each slice's blocks in column order,
// the slices in order): L_k = sum over blocks in order, the first argmin, and
// s* = s_k* from this search's scale table.  With slices that start on
// 256-column boundaries the blocks are the ones one search of the whole
// layer forms, and the sums are the same to the last bit.
__global__ void __launch_bounds__(kRedThreads)
    select_losses_kernel(const double* __restrict__ blk, int64_t nb, int G, double* __restrict__ losses,
                         int32_t* __restrict__ best_idx, const float* __restrict__ s_tab, int64_t D_in,
                         float* __restrict__ s_star, uint32_t* status) {
  __shared__ double sh[kMaxGrid];
  __shared__ int kbest;
  if (threadIdx.x < G) {
    double L = 0.0;
    for (int64_t b = 0; b < nb; ++b) L += blk[static_cast<int64_t>(threadIdx.x) * nb + b];
    sh[threadIdx.x] = L;
    losses[threadIdx.x] = L;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int b = -1;
    double bl = 0.0;
    for (int kk = 0; kk < G; ++kk) {
      const double L = sh[kk];
      if (isnan(L)) continue;
      if (b < 0 || L < bl) {
        b = kk;
        bl = L;
      }
    }
    if (b < 0) {
      b = 0;
      set_error(status, AWQ_DEV_NONFINITE);
    }
    kbest = b;
    *best_idx = b;
  }
  __syncthreads();
  const float* src = s_tab + static_cast<int64_t>(kbest) * D_in;
  for (int64_t j = threadIdx.x; j < D_in; j += kRedThreads) s_star[j] = src[j];
}

cudaError_t launch_select_losses(const double* blk, int64_t nb, int G, double* losses, int32_t* best_idx,
                                 const float* s_tab, int64_t D_in, float* s_star, uint32_t* status,
                                 cudaStream_t stream) {
  select_losses_kernel<<<1, kRedThreads, 0, stream>>>(blk, nb, G, losses, best_idx, s_tab, D_in, s_star, status);
  return cudaGetLastError();
}

int reduce_blocks(int64_t D_out) { return static_cast<int>((D_out + kRedBlockCols - 1) / kRedBlockCols); }

cudaError_t launch_reduce_losses(const float* partial, int m_tiles, int64_t D_out, int G, double* col_losses,
                                 double* blk, unsigned int* ticket, double* losses, int32_t* best_idx,
                                 const float* s_tab, int64_t D_in, float* s_star, uint32_t* status,
                                 cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(reduce_blocks(D_out)), static_cast<unsigned>(G));
  static_assert(kMaxGrid <= kRedSumThreads, "one thread per candidate in the final sums");
  reduce_losses_kernel<<<grid, kRedSumThreads, 0, stream>>>(partial, m_tiles, D_out, G, col_losses, blk, ticket, losses,
                                                         best_idx, s_tab, D_in, s_star, status);
  return cudaGetLastError();
}

}  // namespace awqdev
