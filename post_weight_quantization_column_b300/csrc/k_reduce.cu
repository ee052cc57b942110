// Loss reduction and argmin ("AWQ (Activation-aware Weight Quantization)",
// 缩放因子优化的完整流程 steps 4c-6): the search leaves one fp32 sum of squares
// per (candidate, row tile, column); these are summed in a fixed order, first
// over row tiles (per-column losses), then over columns (L_k, fp64), then
// k* = first argmin and s* = s_k* is copied out.
#include "internal.h"
#include "ptx.cuh"

namespace awqdev {

constexpr int kRedThreads = 256;

// One kernel for the whole reduction.  CTA (bx, k) owns columns
// [256 bx, 256 bx + 256) of candidate k: each thread sums its column over the
// row tiles into col[k][n] -- each run of 8 tiles as a fixed fp32 pairwise
// tree (error below 3 * 2^-24 of the run's sum of squares), the runs in tile
// order in fp64, which keeps fp64 adds (slow on this part) to one per 8
// tiles; the CTA then sums its 256 columns in a fixed fp64 tree into
// blk[k][bx].  The last CTA to finish (a ticket
// counter that the caller zeroed) adds blk[k][0..nb) in block order into
// L_k, picks k* = first argmin and copies s* = s_k*.  Every sum has a fixed
// order, so the result does not depend on timing.
__global__ void __launch_bounds__(kRedThreads)
    reduce_losses_kernel(const float* __restrict__ partial, int m_tiles, int64_t D_out, int G,
                         double* __restrict__ col, double* __restrict__ blk, unsigned int* __restrict__ ticket,
                         double* __restrict__ losses, int32_t* __restrict__ best_idx, const float* __restrict__ s_tab,
                         int64_t D_in, float* __restrict__ s_star, uint32_t* status) {
  __shared__ double sh[kRedThreads];
  __shared__ bool last;
  __shared__ int kbest;
  const int k = blockIdx.y;
  const int nb = gridDim.x;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * kRedThreads + threadIdx.x;
  double v = 0.0;
  if (n < D_out) {
    const float* p = partial + static_cast<int64_t>(k) * m_tiles * D_out + n;
    for (int m = 0; m < m_tiles; m += 8) {
      float x[8];  // eight loads in flight; tiles past the end count as 0
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = m + i < m_tiles ? p[static_cast<int64_t>(m + i) * D_out] : 0.f;
      const float t = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
      v += static_cast<double>(t);
    }
    col[static_cast<int64_t>(k) * D_out + n] = v;
  }
  sh[threadIdx.x] = v;
  __syncthreads();
  for (int w = kRedThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    blk[static_cast<int64_t>(k) * nb + blockIdx.x] = sh[0];
    __threadfence();
    const unsigned int done = atomicAdd(ticket, 1u);
    last = done == static_cast<unsigned int>(nb) * static_cast<unsigned int>(G) - 1u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x < G) {
    double L = 0.0;
#pragma unroll 4
    for (int b = 0; b < nb; ++b) L += blk[static_cast<int64_t>(threadIdx.x) * nb + b];
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
    *ticket = 0u;  // ready for the next call on this workspace
  }
  __syncthreads();
  const float* src = s_tab + static_cast<int64_t>(kbest) * D_in;
  if ((reinterpret_cast<uintptr_t>(s_star) & 15u) == 0 && (D_in & 3) == 0) {
    // s_tab rows start 16-byte aligned (D_in is a multiple of the group size)
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* d4 = reinterpret_cast<float4*>(s_star);
#pragma unroll 4
    for (int64_t j = threadIdx.x; j < D_in / 4; j += kRedThreads) d4[j] = s4[j];
  } else {
    for (int64_t j = threadIdx.x; j < D_in; j += kRedThreads) s_star[j] = src[j];
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

int reduce_blocks(int64_t D_out) { return static_cast<int>((D_out + kRedThreads - 1) / kRedThreads); }

cudaError_t launch_reduce_losses(const float* partial, int m_tiles, int64_t D_out, int G, double* col_losses,
                                 double* blk, unsigned int* ticket, double* losses, int32_t* best_idx,
                                 const float* s_tab, int64_t D_in, float* s_star, uint32_t* status,
                                 cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(reduce_blocks(D_out)), static_cast<unsigned>(G));
  reduce_losses_kernel<<<grid, kRedThreads, 0, stream>>>(partial, m_tiles, D_out, G, col_losses, blk, ticket, losses,
                                                         best_idx, s_tab, D_in, s_star, status);
  return cudaGetLastError();
}

}  // namespace awqdev
