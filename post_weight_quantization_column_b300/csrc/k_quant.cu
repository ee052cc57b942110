// Scale table, per-group quantiser parameters, candidate materialisation and
// the bit-exact int4 pack.
//
// Quantiser ("AWQ (Activation-aware Weight Quantization)", 技术原理 -
// 量化数学基础; aiqz.cc article "awq-activation-aware-quantization", section 4;
// asymmetric zero-point form of the CSDN AutoAWQ walkthrough's quant_config):
//   asymmetric: step = fp16((max(w',0) - min(w',0)) / 15), zero = clamp(rint(-min/step), 0, 15),
//               code = clamp(rint(w'/step) + zero, 0, 15)
//   symmetric:  step = fp16(max|w'| / 7), code = clamp(rint(w'/step), -7, 7) (+8 when stored)
//   dequant (code - zero) * step; a zero step gives dequant 0.
// The pack reproduces the IEEE fp32 round-to-nearest quotient w'/step exactly;
// the search uses a reciprocal multiply (its loss tolerance allows it).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {

// 1.5 * 2^23: adding it to |x| < 2^22 rounds x to an integer (ties to even)
// held in the low mantissa bits.
constexpr float kMagic = 12582912.0f;

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ bool bf16x2_nonfinite(uint32_t u) {
  return ((u & 0x7F80u) == 0x7F80u) || ((u & 0x7F800000u) == 0x7F800000u);
}

// ------------------------------------------------------------------ scales
// s_kj = fp32(pow(fp64(max(a_j, floor)), alpha_k)), r_kj = 1/s_kj (IEEE).
// "AWQ (Activation-aware Weight Quantization)", 缩放因子优化的完整流程 step 3.
__global__ void scale_table_kernel(const float* __restrict__ mean_abs, int64_t D, AlphaGrid grid, float act_floor,
                                   float* __restrict__ s_tab, float* __restrict__ r_tab, uint32_t* status) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int k = blockIdx.y;
  if (j >= D) return;
  const float a = mean_abs[j];
  if (!isfinite(a) && k == 0) set_error(status, AWQ_DEV_NONFINITE);
  const float af = fmaxf(a, act_floor);
  const float s = static_cast<float>(pow(static_cast<double>(af), grid.a[k]));
  s_tab[static_cast<int64_t>(k) * D + j] = s;
  r_tab[static_cast<int64_t>(k) * D + j] = __fdiv_rn(1.0f, s);
}

cudaError_t launch_scale_table(const float* mean_abs, int64_t D_in, const AlphaGrid& grid, int G, float act_floor,
                               float* s_tab, float* r_tab, uint32_t* status, cudaStream_t stream) {
  const dim3 g(static_cast<unsigned>((D_in + 255) / 256), static_cast<unsigned>(G));
  scale_table_kernel<<<g, 256, 0, stream>>>(mean_abs, D_in, grid, act_floor, s_tab, r_tab, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ group parameters
// Exact step / zero of one (group, column) from the range of its scaled weights.
__device__ __forceinline__ QParam make_qparam(float lo, float hi, int symmetric, uint32_t* status) {
  QParam q;
  q.pad = 0.f;
  const float raw = symmetric ? __fdiv_rn(hi, 7.0f) : __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
  float sc = __half2float(__float2half_rn(raw));
  if (isinf(sc)) {
    set_error(status, AWQ_DEV_RANGE);
    sc = 0.f;
  }
  if (sc == 0.f) {
    q.inv = 0.f;
    q.zm = kMagic;
    q.step = 0.f;
    return q;
  }
  float z = 0.f;
  // an integer code in [0, 15]; the int round trip also turns -0 into +0
  if (!symmetric) z = static_cast<float>(static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(-lo, sc)), 0.f), 15.f)));
  q.inv = __frcp_rn(sc);
  q.zm = kMagic + z;
  q.step = sc;
  return q;
}

// Running min / max of three values (sm_100 three-input forms; exact, so the
// order of the comparisons does not matter).
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// max(|a|, |b|, |c|)
__device__ __forceinline__ float fmaxabs3(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

constexpr int kGpThreads = 128;   // one output column per thread
constexpr int kGpCols = kGpThreads;
constexpr int kMaxGpCandidates = 32;  // candidates per CTA (grid.z splits larger grids)

// One CTA: one group of GS rows x 128 columns, up to 32 candidates.  The W tile
// (GS x 128 bf16) and the group's scale rows sit in shared memory, the
// scales as {s_k[r], s_k[r+1]} pairs so that one 8-byte broadcast load feeds
// a packed multiply.  Thread t owns column t and keeps the running range of
// all G candidates in registers: for each pair of rows it unpacks its two
// weights once, then per candidate does w' = w s for both rows in one packed
// multiply and a three-input min / max against the running range.
template <int GS>
__global__ void __launch_bounds__(kGpThreads) group_params_kernel(const __nv_bfloat16* __restrict__ W,
                                                                const float* __restrict__ s_tab, int64_t D_in,
                                                                int64_t D_out, int G, int symmetric,
                                                                float* __restrict__ qp, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* wsh = reinterpret_cast<__nv_bfloat16*>(smem);     // [GS][128]
  float2* ssh = reinterpret_cast<float2*>(smem + GS * kGpCols * 2);  // [GS/2][nk]
  const int t = threadIdx.x;
  const int k0 = blockIdx.z * kMaxGpCandidates;
  const int nk = min(kMaxGpCandidates, G - k0);
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kGpCols;
  const int64_t grp = blockIdx.y;
  const int64_t j0 = grp * GS;
  bool bad = false;
  {
    // all of the thread's loads in flight before the first store
    constexpr int kLoads = GS * (kGpCols / 8) / kGpThreads;
    uint4 v[kLoads];
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const int idx = t + i * kGpThreads;
      const int64_t col = n0 + (idx & 15) * 8;
      v[i] = col < D_out ? *reinterpret_cast<const uint4*>(W + (j0 + (idx >> 4)) * D_out + col)
                         : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const int idx = t + i * kGpThreads;
      bad |= bf16x2_nonfinite(v[i].x) | bf16x2_nonfinite(v[i].y) | bf16x2_nonfinite(v[i].z) |
             bf16x2_nonfinite(v[i].w);
      *reinterpret_cast<uint4*>(wsh + (idx >> 4) * kGpCols + (idx & 15) * 8) = v[i];
    }
  }
  {
    // scale pairs, up to kMaxGpCandidates * GS/2 of them: all loads first
    constexpr int kSLoads = kMaxGpCandidates * (GS / 2) / kGpThreads;
    float2 sv[kSLoads];
#pragma unroll
    for (int i = 0; i < kSLoads; ++i) {
      const int idx = t + i * kGpThreads;
      const int k = idx / (GS / 2);
      const int rp = idx - k * (GS / 2);
      sv[i] = k < nk ? *reinterpret_cast<const float2*>(s_tab + static_cast<int64_t>(k0 + k) * D_in + j0 + 2 * rp)
                     : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kSLoads; ++i) {
      const int idx = t + i * kGpThreads;
      const int k = idx / (GS / 2);
      const int rp = idx - k * (GS / 2);
      if (k < nk) ssh[rp * nk + k] = sv[i];
    }
  }
  if (bad && blockIdx.z == 0) set_error(status, AWQ_DEV_NONFINITE);
  __syncthreads();
  const int64_t n = n0 + t;
  if (n >= D_out) return;

  float lo[kMaxGpCandidates], hi[kMaxGpCandidates];
#pragma unroll
  for (int k = 0; k < kMaxGpCandidates; ++k) lo[k] = hi[k] = 0.f;
  const uint16_t* wcol = reinterpret_cast<const uint16_t*>(wsh) + t;
#pragma unroll 2
  for (int rp = 0; rp < GS / 2; ++rp) {
    const float2 w2 = make_float2(__uint_as_float(static_cast<uint32_t>(wcol[(2 * rp) * kGpCols]) << 16),
                                  __uint_as_float(static_cast<uint32_t>(wcol[(2 * rp + 1) * kGpCols]) << 16));
    const float2* sp = ssh + rp * nk;
    if (symmetric) {
#pragma unroll
      for (int k = 0; k < kMaxGpCandidates; ++k) {
        if (k < nk) {
          const float2 p = __fmul2_rn(w2, sp[k]);
          hi[k] = fmaxabs3(hi[k], p.x, p.y);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < kMaxGpCandidates; ++k) {
        if (k < nk) {
          const float2 p = __fmul2_rn(w2, sp[k]);
          lo[k] = fmin3(lo[k], p.x, p.y);
          hi[k] = fmax3(hi[k], p.x, p.y);
        }
      }
    }
  }
  const int64_t T = D_in / GS;
  const int64_t kstride = T * (D_out / kQChunkCols) * kQChunkFloats;
  float* dst0 = qp + k0 * kstride + (grp * (D_out / kQChunkCols) + n / kQChunkCols) * kQChunkFloats +
                (n % kQChunkCols);
#pragma unroll
  for (int k = 0; k < kMaxGpCandidates; ++k) {
    if (k < nk) {
      const QParam q = make_qparam(lo[k], hi[k], symmetric, status);
      float* dst = dst0 + k * kstride;
      dst[0] = q.inv;
      dst[kQChunkCols] = q.zm;
      dst[2 * kQChunkCols] = q.step;
    }
  }
}

static size_t group_params_smem(int GS) {
  return static_cast<size_t>(GS) * kGpCols * 2 + static_cast<size_t>(GS / 2) * kMaxGpCandidates * 8;
}

template <int GS>
static cudaError_t launch_group_params_t(const __nv_bfloat16* W, const float* s_tab, int64_t D_in, int64_t D_out,
                                         int G, int symmetric, float* qp, uint32_t* status, cudaStream_t stream) {
  const size_t smem = group_params_smem(GS);
  cudaError_t e = cudaFuncSetAttribute(group_params_kernel<GS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((D_out + kGpCols - 1) / kGpCols), static_cast<unsigned>(D_in / GS),
                  static_cast<unsigned>((G + kMaxGpCandidates - 1) / kMaxGpCandidates));
  group_params_kernel<GS><<<grid, kGpThreads, smem, stream>>>(W, s_tab, D_in, D_out, G, symmetric, qp, status);
  return cudaGetLastError();
}

cudaError_t launch_group_params(const void* W, const float* s_tab, int64_t D_in, int64_t D_out, int G,
                                int group_size, int symmetric, float* qp, uint32_t* status, cudaStream_t stream) {
  const __nv_bfloat16* Wb = static_cast<const __nv_bfloat16*>(W);
  switch (group_size) {
    case 64:
      return launch_group_params_t<64>(Wb, s_tab, D_in, D_out, G, symmetric, qp, status, stream);
    case 128:
      return launch_group_params_t<128>(Wb, s_tab, D_in, D_out, G, symmetric, qp, status, stream);
    case 256:
      return launch_group_params_t<256>(Wb, s_tab, D_in, D_out, G, symmetric, qp, status, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------------ candidate materialisation
// dW_k[j, n] = bf16( (code - zero) * step / s_kj - w_jn ): the difference form
// S^-1 W'hat - W of one candidate, so that X * dW_k is the output error of
// "AWQ (Activation-aware Weight Quantization)", 缩放因子优化的完整流程 step 4c.
__device__ __forceinline__ float dq_delta(float w, float s, float r, const QParam& q, float lo, float hi) {
  const float wp = w * s;
  float t = fmaf(wp, q.inv, q.zm);
  t = fminf(fmaxf(t, lo), hi);
  const float d = (t - q.zm) * q.step;
  return fmaf(d, r, -w);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(256) materialize_kernel(const __nv_bfloat16* __restrict__ W,
                                                        const float* __restrict__ s_tab,
                                                        const float* __restrict__ r_tab,
                                                        const float* __restrict__ qp, int64_t D_in, int64_t D_out,
                                                        int group_size, float lo, float hi,
                                                        __nv_bfloat16* __restrict__ dW) {
  const int lane = threadIdx.x & 31;
  const int rl = threadIdx.x >> 5;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 256 + lane * 8;
  if (n >= D_out) return;
  const int k = blockIdx.z;
  const int64_t jb = static_cast<int64_t>(blockIdx.y) * 64;
  const int64_t T = D_in / group_size;
  const int64_t grp = jb / group_size;
  const float* q = qp + ((static_cast<int64_t>(k) * T + grp) * (D_out / kQChunkCols) + n / kQChunkCols) * kQChunkFloats;
  QParam qv[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) qv[c] = QParam{q[c], q[kQChunkCols + c], q[2 * kQChunkCols + c], 0.f};
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const int64_t j = jb + rl + 8 * i;
    const float s = s_tab[static_cast<int64_t>(k) * D_in + j];
    const float r = r_tab[static_cast<int64_t>(k) * D_in + j];
    const uint4 wv = *reinterpret_cast<const uint4*>(W + j * D_out + n);
    const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
    uint32_t o[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float d0 = dq_delta(bf16lo(wu[c]), s, r, qv[2 * c], lo, hi);
      const float d1 = dq_delta(bf16hi(wu[c]), s, r, qv[2 * c + 1], lo, hi);
      o[c] = pack_bf16x2(d0, d1);
    }
    *reinterpret_cast<uint4*>(dW + (static_cast<int64_t>(k) * D_in + j) * D_out + n) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_materialize(const void* W, const float* s_tab, const float* r_tab, const float* qp,
                               int64_t D_in, int64_t D_out, int G, int group_size, int symmetric, void* dW,
                               cudaStream_t stream) {
  const float lo = symmetric ? kMagic - 7.f : kMagic;
  const float hi = symmetric ? kMagic + 7.f : kMagic + 15.f;
  const dim3 grid(static_cast<unsigned>((D_out + 255) / 256), static_cast<unsigned>(D_in / 64),
                  static_cast<unsigned>(G));
  materialize_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(W), s_tab, r_tab, qp, D_in, D_out,
                                               group_size, lo, hi, static_cast<__nv_bfloat16*>(dW));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ pack
// "AWQ (Activation-aware Weight Quantization)", 推理时的等效实现:
// W_quantized = Quantize(diag(s*) W); "009. AWQ Integration", Consequences:
// two 4-bit codes per byte (even input row in the low nibble).
//
// One CTA: one group (GS rows) x 64 columns, 256 threads.  Thread t owns the
// 8 columns of chunk c = t % 8 and the row pairs (2p + 64i, 2p + 64i + 1),
// p = t / 8, i < GS/64, so that both rows of a packed byte sit in one
// thread.  Pass 1 finds the per-column range (shuffles over the 4 row slots
// of a warp, then the 8 warps in a fixed order in shared memory) and the
// exact step / zero; pass 2 emits codes.
//
// Codes equal clamp(rint(fp32(w'/step)) + zero): the quotient is first
// formed as w' * (1/step); where that lands within 8e-6 of a half-integer
// (where the two could round differently), the thread redoes its rows with
// the IEEE division.  |w'/step| <= 45 in every case, where the product is
// within 6e-6 of the IEEE quotient, so elsewhere both round alike.
constexpr float kTieGuard = 0.5f - 8.0e-6f;
constexpr int kPackCols = 64;

template <int GS>
__global__ void __launch_bounds__(256) pack_kernel(const __nv_bfloat16* __restrict__ W, const float* __restrict__ s,
                                                 int64_t D_in, int64_t D_out, int symmetric,
                                                 uint8_t* __restrict__ qweight, __half* __restrict__ scales,
                                                 __half* __restrict__ zeros, uint32_t* status) {
  constexpr int NP = GS / 64;  // row pairs per thread
  constexpr int NR = 2 * NP;   // rows per thread
  __shared__ float red_lo[8][kPackCols];
  __shared__ float red_hi[8][kPackCols];
  __shared__ float4 prm[kPackCols];  // {step, 1/step, zoff, zero}
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int wp_ = t >> 5;
  const int c = t & 7;
  const int pslot = t >> 3;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * kPackCols + c * 8;
  const int64_t grp = blockIdx.y;
  const int64_t jb = grp * GS + 2 * pslot;  // row pair i: jb + 64 i, jb + 64 i + 1
  const bool active = n < D_out;

  uint4 w[NR];
  float sj[NR];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int64_t row = jb + 64 * (i >> 1) + (i & 1);
    sj[i] = s[row];
    w[i] = active ? *reinterpret_cast<const uint4*>(W + row * D_out + n) : make_uint4(0u, 0u, 0u, 0u);
    bad |= bf16x2_nonfinite(w[i].x) | bf16x2_nonfinite(w[i].y) | bf16x2_nonfinite(w[i].z) | bf16x2_nonfinite(w[i].w);
  }
  if (bad) set_error(status, AWQ_DEV_NONFINITE);

  // pass 1: per-column range of w' = w * s over this thread's rows (two rows
  // per step: packed products, three-input min / max)
  float lo[8], hi[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) lo[k] = hi[k] = 0.f;
#pragma unroll
  for (int i = 0; i < NR; i += 2) {
    const uint32_t we[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
    const uint32_t wo[4] = {w[i + 1].x, w[i + 1].y, w[i + 1].z, w[i + 1].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 pe = __fmul2_rn(make_float2(bf16lo(we[k]), bf16hi(we[k])), make_float2(sj[i], sj[i]));
      const float2 po = __fmul2_rn(make_float2(bf16lo(wo[k]), bf16hi(wo[k])), make_float2(sj[i + 1], sj[i + 1]));
      if (symmetric) {
        hi[2 * k] = fmaxabs3(hi[2 * k], pe.x, po.x);
        hi[2 * k + 1] = fmaxabs3(hi[2 * k + 1], pe.y, po.y);
      } else {
        lo[2 * k] = fmin3(lo[2 * k], pe.x, po.x);
        hi[2 * k] = fmax3(hi[2 * k], pe.x, po.x);
        lo[2 * k + 1] = fmin3(lo[2 * k + 1], pe.y, po.y);
        hi[2 * k + 1] = fmax3(hi[2 * k + 1], pe.y, po.y);
      }
    }
  }
  // lanes l, l^8, l^16, l^24 hold the same columns (four row slots)
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    lo[k] = fminf(lo[k], __shfl_xor_sync(0xFFFFFFFFu, lo[k], 8));
    hi[k] = fmaxf(hi[k], __shfl_xor_sync(0xFFFFFFFFu, hi[k], 8));
    lo[k] = fminf(lo[k], __shfl_xor_sync(0xFFFFFFFFu, lo[k], 16));
    hi[k] = fmaxf(hi[k], __shfl_xor_sync(0xFFFFFFFFu, hi[k], 16));
  }
  if (lane < 8) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      red_lo[wp_][c * 8 + k] = lo[k];
      red_hi[wp_][c * 8 + k] = hi[k];
    }
  }
  __syncthreads();
  if (t < kPackCols) {
    const int col = t;
    float l = 0.f, h = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      l = fminf(l, red_lo[k][col]);
      h = fmaxf(h, red_hi[k][col]);
    }
    const float raw = symmetric ? __fdiv_rn(h, 7.0f) : __fdiv_rn(__fsub_rn(h, l), 15.0f);
    float sc = __half2float(__float2half_rn(raw));
    if (isinf(sc)) {
      set_error(status, AWQ_DEV_RANGE);
      sc = 0.f;
    }
    float z = 0.f;
    if (!symmetric && sc != 0.f)
      z = static_cast<float>(static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(-l, sc)), 0.f), 15.f)));
    const float zoff = symmetric ? 8.f : z;
    prm[col] = make_float4(sc, sc != 0.f ? __frcp_rn(sc) : 0.f, zoff, symmetric ? 8.f : z);
    const int64_t ncol = static_cast<int64_t>(blockIdx.x) * kPackCols + col;
    if (ncol < D_out) {
      scales[grp * D_out + ncol] = __float2half_rn(sc);
      zeros[grp * D_out + ncol] = __float2half_rn(symmetric ? 8.f : z);
    }
  }
  __syncthreads();
  if (!active) return;

  float step[8], inv[8], zmz[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float4 pr = prm[c * 8 + k];
    step[k] = pr.x;
    inv[k] = pr.y;
    zmz[k] = kMagic + pr.z;
  }
  const float clo = symmetric ? kMagic + 1.f : kMagic;
  const float chi = kMagic + 15.f;

  // pass 2 (fast): codes through the reciprocal.  y = w' (1/step); c =
  // y + 1.5*2^23 + zero rounds it to an integer; tmax tracks the largest
  // |y - rint(y)|, which flags a near tie anywhere in the thread's elements.
  uint32_t out[NP][2];
  float tmax = 0.f;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const uint32_t we[4] = {w[2 * i].x, w[2 * i].y, w[2 * i].z, w[2 * i].w};
    const uint32_t wo[4] = {w[2 * i + 1].x, w[2 * i + 1].y, w[2 * i + 1].z, w[2 * i + 1].w};
    uint32_t bytes[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 inv2 = make_float2(inv[2 * k], inv[2 * k + 1]);
      const float2 zm2 = make_float2(zmz[2 * k], zmz[2 * k + 1]);
      const float2 nzm2 = make_float2(-zmz[2 * k], -zmz[2 * k + 1]);
      const float2 ye = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(we[k]), bf16hi(we[k])), make_float2(sj[2 * i], sj[2 * i])), inv2);
      const float2 yo = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(wo[k]), bf16hi(wo[k])), make_float2(sj[2 * i + 1], sj[2 * i + 1])), inv2);
      float2 ce = __fadd2_rn(ye, zm2);
      float2 co = __fadd2_rn(yo, zm2);
      const float2 de = __ffma2_rn(ye, make_float2(-1.f, -1.f), __fadd2_rn(ce, nzm2));
      const float2 dd = __ffma2_rn(yo, make_float2(-1.f, -1.f), __fadd2_rn(co, nzm2));
      tmax = fmaxabs3(tmax, de.x, de.y);
      tmax = fmaxabs3(tmax, dd.x, dd.y);
      ce.x = fminf(fmaxf(ce.x, clo), chi);
      ce.y = fminf(fmaxf(ce.y, clo), chi);
      co.x = fminf(fmaxf(co.x, clo), chi);
      co.y = fminf(fmaxf(co.y, clo), chi);
      bytes[2 * k] = (__float_as_uint(ce.x) & 0xFu) | ((__float_as_uint(co.x) & 0xFu) << 4);
      bytes[2 * k + 1] = (__float_as_uint(ce.y) & 0xFu) | ((__float_as_uint(co.y) & 0xFu) << 4);
    }
    out[i][0] = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
    out[i][1] = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
  }
  const bool tie = tmax > kTieGuard;
  if (tie) {
    // slow path: IEEE quotient for every element of this thread
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const uint32_t we[4] = {w[2 * i].x, w[2 * i].y, w[2 * i].z, w[2 * i].w};
      const uint32_t wo[4] = {w[2 * i + 1].x, w[2 * i + 1].y, w[2 * i + 1].z, w[2 * i + 1].w};
      uint32_t bytes[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float xe = (k & 1) ? bf16hi(we[k >> 1]) : bf16lo(we[k >> 1]);
        const float xo = (k & 1) ? bf16hi(wo[k >> 1]) : bf16lo(wo[k >> 1]);
        // clamp(rint(IEEE w'/step) + zoff, clo, 15); a zero step keeps code zoff
        uint32_t ke = static_cast<uint32_t>(zmz[k] - kMagic), ko = ke;
        if (step[k] != 0.f) {
          const float zo = zmz[k] - kMagic;
          const float ql = clo - kMagic;
          const float qe = rintf(__fdiv_rn(__fmul_rn(xe, sj[2 * i]), step[k])) + zo;
          const float qo = rintf(__fdiv_rn(__fmul_rn(xo, sj[2 * i + 1]), step[k])) + zo;
          ke = static_cast<uint32_t>(fminf(fmaxf(qe, ql), 15.f));
          ko = static_cast<uint32_t>(fminf(fmaxf(qo, ql), 15.f));
        }
        bytes[k] = ke | (ko << 4);
      }
      out[i][0] = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
      out[i][1] = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
    }
  }
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int64_t prow = (jb + 64 * i) / 2;
    *reinterpret_cast<uint2*>(qweight + prow * D_out + n) = make_uint2(out[i][0], out[i][1]);
  }
}

cudaError_t launch_pack(const void* W, const float* s, int64_t D_in, int64_t D_out, int group_size, int symmetric,
                        uint8_t* qweight, void* scales, void* zeros, uint32_t* status, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((D_out + kPackCols - 1) / kPackCols), static_cast<unsigned>(D_in / group_size));
  const __nv_bfloat16* Wb = static_cast<const __nv_bfloat16*>(W);
  __half* sc = static_cast<__half*>(scales);
  __half* zr = static_cast<__half*>(zeros);
  switch (group_size) {
    case 64:
      pack_kernel<64><<<grid, 256, 0, stream>>>(Wb, s, D_in, D_out, symmetric, qweight, sc, zr, status);
      break;
    case 128:
      pack_kernel<128><<<grid, 256, 0, stream>>>(Wb, s, D_in, D_out, symmetric, qweight, sc, zr, status);
      break;
    case 256:
      pack_kernel<256><<<grid, 256, 0, stream>>>(Wb, s, D_in, D_out, symmetric, qweight, sc, zr, status);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace awqdev
