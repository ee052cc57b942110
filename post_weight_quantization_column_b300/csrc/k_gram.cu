// The Gram form of the search loss.  With H = X^T X and a factor H = L L^T
// (Cholesky, L lower triangular), every candidate's loss
//   L_k = ||X D_k||^2 = sum_n d_n^T H d_n = ||L^T D_k||^2
// so the fused search run on R = L^T (D_in rows) in place of X (N rows) gives
// the same losses with D_in / N of the flops.  This file holds the steps that
// build R: a tiled transpose of X (so that the tensor-core GEMM can form
// X^T X from a K-major operand), a right-looking blocked Cholesky in fp32
// (64 x 64 blocks: the diagonal block factored in shared memory together
// with its triangular inverse, the panel below it as a product with that
// inverse, the trailing lower triangle updated by a register-tiled product),
// and the transposed conversion of L to bf16 R.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {
namespace {

constexpr int kCb = 64;  // Cholesky block

// Xt [D, ldt] (row j = channel j, the N rows of X along it, zero past N)
__global__ void transpose_x_kernel(const __nv_bfloat16* __restrict__ X, int64_t N, int64_t D, int64_t ldt,
                                   __nv_bfloat16* __restrict__ Xt) {
  __shared__ __nv_bfloat16 tile[32][34];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;  // rows of X (columns of Xt)
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * 32;  // channels
  const int tx = threadIdx.x, ty = threadIdx.y;              // 32 x 8
  for (int i = ty; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    tile[i][tx] = (r < N && c < D) ? X[r * D + c] : __float2bfloat16(0.f);
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (c < D && r < ldt) Xt[c * ldt + r] = tile[tx][i];
  }
}

// Factor the diagonal block (k, k) in place, A_kk = L_kk L_kk^T, and write
// the inverse of L_kk (lower triangular, zeros above) to Linv.  Per column j
// of the block: every thread reads the pivot, the column below it is scaled
// (barrier), the trailing lower triangle is updated by a 16 x 16 thread grid
// (barrier).  The diagonal of L goes to a separate array so that the pivot
// the threads read is never overwritten inside a step.  The inverse is
// formed by one thread per column (forward substitution on the identity).
__global__ void __launch_bounds__(256) chol_diag_kernel(float* __restrict__ A, int64_t D, int k,
                                                        float* __restrict__ Linv, uint32_t* status) {
  __shared__ float S[kCb][kCb + 1];
  __shared__ float Li[kCb][kCb + 1];
  __shared__ float Ld[kCb];
  const int t = threadIdx.x;
  const int ty = t / 16, tx = t % 16;
  const int64_t o = static_cast<int64_t>(k) * kCb;
  for (int i = t; i < kCb * kCb; i += 256) S[i / kCb][i % kCb] = A[(o + i / kCb) * D + o + i % kCb];
  __syncthreads();
  for (int j = 0; j < kCb; ++j) {
    float d = S[j][j];
    if (!(d > 0.f) || !isfinite(d)) {
      if (t == 0) set_error(status, AWQ_DEV_RANGE);  // not positive definite
      d = 1.f;
    }
    const float ljj = __fsqrt_rn(d);
    if (t == 0) Ld[j] = ljj;
    if (t > j && t < kCb) S[t][j] = __fdiv_rn(S[t][j], ljj);
    __syncthreads();
    for (int i = j + 1 + ty; i < kCb; i += 16) {
      const float sij = S[i][j];
      for (int c = j + 1 + tx; c <= i; c += 16) S[i][c] = fmaf(-sij, S[c][j], S[i][c]);
    }
    __syncthreads();
  }
  for (int i = t; i < kCb * kCb; i += 256) {
    const int r = i / kCb, c = i % kCb;
    if (c < r) A[(o + r) * D + o + c] = S[r][c];
    if (c == r) A[(o + r) * D + o + c] = Ld[r];
  }
  if (t < kCb) {
    const int m = t;  // column m of L^-1: rows m .. 63
    for (int r = 0; r < kCb; ++r) {
      float v = r == m ? 1.f : 0.f;
      if (r > m)
        for (int c = m; c < r; ++c) v = fmaf(-S[r][c], Li[c][m], v);
      Li[r][m] = r < m ? 0.f : __fdiv_rn(v, Ld[r]);
    }
  }
  __syncthreads();
  for (int i = t; i < kCb * kCb; i += 256) Linv[i] = Li[i / kCb][i % kCb];
}

// Panel below block k: X L_kk^T = A[rows, block k], i.e. X = A L_kk^-T:
// X[r][j] = sum_{c <= j} A[r][c] Linv[j][c], 64 rows x 64 columns per CTA,
// 4 x 4 outputs per thread, read from shared memory before any is written.
__global__ void __launch_bounds__(256) chol_panel_kernel(float* __restrict__ A, int64_t D, int k,
                                                         const float* __restrict__ Linv) {
  __shared__ float P[kCb][kCb + 1];
  __shared__ float Li[kCb][kCb + 1];
  const int t = threadIdx.x;
  const int64_t o = static_cast<int64_t>(k) * kCb;
  const int64_t r0 = o + kCb + static_cast<int64_t>(blockIdx.x) * kCb;
  for (int e = t; e < kCb * kCb / 4; e += 256) {
    const int r = e / (kCb / 4), c4 = (e % (kCb / 4)) * 4;
    const float4 v = *reinterpret_cast<const float4*>(A + (r0 + r) * D + o + c4);
    const float4 w = *reinterpret_cast<const float4*>(Linv + r * kCb + c4);
    P[r][c4] = v.x;
    P[r][c4 + 1] = v.y;
    P[r][c4 + 2] = v.z;
    P[r][c4 + 3] = v.w;
    Li[r][c4] = w.x;
    Li[r][c4 + 1] = w.y;
    Li[r][c4 + 2] = w.z;
    Li[r][c4 + 3] = w.w;
  }
  __syncthreads();
  const int ty = t / 16, tx = t % 16;  // rows 4 ty .. 4 ty + 3, columns tx + 16 b
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
  for (int c = 0; c < kCb; ++c) {
    float pr[4], lj[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) pr[a] = P[4 * ty + a][c];
#pragma unroll
    for (int b = 0; b < 4; ++b) lj[b] = Li[tx + 16 * b][c];  // zero for c > j
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(pr[a], lj[b], acc[a][b]);
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) A[(r0 + 4 * ty + a) * D + o + tx + 16 * b] = acc[a][b];
}

// Trailing update after block k: A[I, J] -= P_I P_J^T for the lower block
// tiles (I >= J) of the trailing matrix, P = the panel of block column k.
__global__ void __launch_bounds__(256) chol_update_kernel(float* __restrict__ A, int64_t D, int k) {
  __shared__ float Pi[kCb][kCb + 1];
  __shared__ float Pj[kCb][kCb + 1];
  // block index -> (I, J), I >= J, over the trailing block rows k+1 ..
  const int64_t tt = blockIdx.x;
  int64_t I = static_cast<int64_t>((sqrt(8.0 * static_cast<double>(tt) + 1.0) - 1.0) / 2.0);
  while (I * (I + 1) / 2 > tt) --I;
  while ((I + 1) * (I + 2) / 2 <= tt) ++I;
  const int64_t J = tt - I * (I + 1) / 2;
  const int64_t o = static_cast<int64_t>(k) * kCb;
  const int64_t ri = o + kCb + I * kCb, rj = o + kCb + J * kCb;
  const int t = threadIdx.x;
  for (int e = t; e < kCb * kCb / 4; e += 256) {
    const int r = e / (kCb / 4), c4 = (e % (kCb / 4)) * 4;
    const float4 vi = *reinterpret_cast<const float4*>(A + (ri + r) * D + o + c4);
    const float4 vj = *reinterpret_cast<const float4*>(A + (rj + r) * D + o + c4);
    Pi[r][c4] = vi.x;
    Pi[r][c4 + 1] = vi.y;
    Pi[r][c4 + 2] = vi.z;
    Pi[r][c4 + 3] = vi.w;
    Pj[r][c4] = vj.x;
    Pj[r][c4 + 1] = vj.y;
    Pj[r][c4 + 2] = vj.z;
    Pj[r][c4 + 3] = vj.w;
  }
  __syncthreads();
  const int ty = t / 16, tx = t % 16;  // rows 4 ty .. 4 ty + 3, columns tx + 16 q
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
  for (int c = 0; c < kCb; ++c) {
    float pi[4], pj[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) pi[a] = Pi[4 * ty + a][c];
#pragma unroll
    for (int b = 0; b < 4; ++b) pj[b] = Pj[tx + 16 * b][c];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(pi[a], pj[b], acc[a][b]);
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t r = ri + 4 * ty + a;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t c = rj + tx + 16 * b;
      if (I != J || c <= r) A[r * D + c] -= acc[a][b];
    }
  }
}

// R = L^T in bf16: R[i, j] = L[j, i] for j >= i, 0 below the diagonal.
__global__ void lt_to_bf16_kernel(const float* __restrict__ L, int64_t D, __nv_bfloat16* __restrict__ R) {
  __shared__ float tile[32][33];
  const int64_t i0 = static_cast<int64_t>(blockIdx.y) * 32;  // rows of R
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * 32;  // columns of R
  const int tx = threadIdx.x, ty = threadIdx.y;              // 32 x 8
  for (int a = ty; a < 32; a += 8) {
    const int64_t j = j0 + a, i = i0 + tx;  // L[j, i]
    tile[a][tx] = (j < D && i < D && j >= i) ? L[j * D + i] : 0.f;
  }
  __syncthreads();
  for (int a = ty; a < 32; a += 8) {
    const int64_t i = i0 + a, j = j0 + tx;
    if (i < D && j < D) R[i * D + j] = __float2bfloat16_rn(tile[tx][a]);
  }
}

}  // namespace

cudaError_t launch_transpose_x(const void* X, int64_t N, int64_t D, int64_t ldt, void* Xt, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((ldt + 31) / 32), static_cast<unsigned>((D + 31) / 32));
  transpose_x_kernel<<<grid, dim3(32, 8), 0, stream>>>(static_cast<const __nv_bfloat16*>(X), N, D, ldt,
                                                        static_cast<__nv_bfloat16*>(Xt));
  return cudaGetLastError();
}

cudaError_t launch_cholesky(float* A, int64_t D, float* Linv, uint32_t* status, cudaStream_t stream) {
  const int nb = static_cast<int>(D / kCb);
  for (int k = 0; k < nb; ++k) {
    chol_diag_kernel<<<1, 256, 0, stream>>>(A, D, k, Linv, status);
    const int rest = nb - k - 1;  // trailing block rows
    if (rest > 0) {
      chol_panel_kernel<<<static_cast<unsigned>(rest), 256, 0, stream>>>(A, D, k, Linv);
      const int64_t tiles = static_cast<int64_t>(rest) * (rest + 1) / 2;
      chol_update_kernel<<<static_cast<unsigned>(tiles), 256, 0, stream>>>(A, D, k);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_lt_to_bf16(const float* L, int64_t D, void* R, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((D + 31) / 32), static_cast<unsigned>((D + 31) / 32));
  lt_to_bf16_kernel<<<grid, dim3(32, 8), 0, stream>>>(L, D, static_cast<__nv_bfloat16*>(R));
  return cudaGetLastError();
}

}  // namespace awqdev
