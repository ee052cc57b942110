// Loss reduction and argmin ("AWQ (Activation-aware Weight Quantization)",
// 缩放因子优化的完整流程 steps 4c-6): the GEMM leaves one fp32 sum of squares
// per (candidate, 128-row tile, column); these are summed in fp64 in a fixed
// order, first over row tiles (per-column losses), then over columns (L_k),
// then k* = first argmin and s* = s_k* is copied out.
#include "internal.h"
#include "ptx.cuh"

namespace awqdev {

__global__ void reduce_rows_kernel(const float* __restrict__ partial, int m_tiles, int64_t D_out,
                                   double* __restrict__ col) {
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int k = blockIdx.y;
  if (n >= D_out) return;
  const float* p = partial + static_cast<int64_t>(k) * m_tiles * D_out + n;
  double s = 0.0;
  for (int m = 0; m < m_tiles; ++m) s += static_cast<double>(p[static_cast<int64_t>(m) * D_out]);
  col[static_cast<int64_t>(k) * D_out + n] = s;
}

constexpr int kRedThreads = 256;

__global__ void __launch_bounds__(kRedThreads) reduce_cols_kernel(const double* __restrict__ col, int64_t D_out,
                                                                 double* __restrict__ losses) {
  __shared__ double sh[kRedThreads];
  const int k = blockIdx.x;
  const double* c = col + static_cast<int64_t>(k) * D_out;
  double s = 0.0;
  for (int64_t n = threadIdx.x; n < D_out; n += kRedThreads) s += c[n];
  sh[threadIdx.x] = s;
  __syncthreads();
  for (int w = kRedThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) losses[k] = sh[0];
}

__global__ void argmin_copy_kernel(const double* __restrict__ losses, int G, const float* __restrict__ s_tab,
                                   int64_t D_in, float* __restrict__ s_star, int32_t* __restrict__ best_idx,
                                   uint32_t* status) {
  __shared__ int kbest;
  if (threadIdx.x == 0) {
    int b = -1;
    double bl = 0.0;
    for (int k = 0; k < G; ++k) {
      const double L = losses[k];
      if (isnan(L)) continue;
      if (b < 0 || L < bl) {
        b = k;
        bl = L;
      }
    }
    if (b < 0) {
      b = 0;
      set_error(status, AWQ_DEV_NONFINITE);
    }
    kbest = b;
    if (blockIdx.x == 0) *best_idx = b;
  }
  __syncthreads();
  const float* src = s_tab + static_cast<int64_t>(kbest) * D_in;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < D_in;
       j += static_cast<int64_t>(gridDim.x) * blockDim.x)
    s_star[j] = src[j];
}

cudaError_t launch_reduce_losses(const float* partial, int m_tiles, int64_t D_out, int G, double* col_losses,
                                 double* losses, int32_t* best_idx, const float* s_tab, int64_t D_in, float* s_star,
                                 uint32_t* status, cudaStream_t stream) {
  const dim3 g1(static_cast<unsigned>((D_out + 255) / 256), static_cast<unsigned>(G));
  reduce_rows_kernel<<<g1, 256, 0, stream>>>(partial, m_tiles, D_out, col_losses);
  reduce_cols_kernel<<<G, kRedThreads, 0, stream>>>(col_losses, D_out, losses);
  unsigned blocks = static_cast<unsigned>((D_in + 1023) / 1024);
  if (blocks < 1) blocks = 1;
  if (blocks > 64) blocks = 64;
  argmin_copy_kernel<<<blocks, 1024, 0, stream>>>(losses, G, s_tab, D_in, s_star, best_idx, status);
  return cudaGetLastError();
}

}  // namespace awqdev
