// Scale table and per-group quantiser parameters of the search (the
// bit-exact int4 pack is in k_pack.cu).
//
// Quantiser ("AWQ (Activation-aware Weight Quantization)", 技术原理 -
// 量化数学基础; aiqz.cc article "awq-activation-aware-quantization", section 4;
// asymmetric zero-point form of the CSDN AutoAWQ walkthrough's quant_config):
//   asymmetric: step = fp16((max(w',0) - min(w',0)) / 15), zero = clamp(rint(-min/step), 0, 15),
//               code = clamp(rint(w'/step) + zero, 0, 15)
//   symmetric:  step = fp16(max|w'| / 7), code = clamp(rint(w'/step), -7, 7) (+8 when stored)
//   dequant (code - zero) * step; a zero step gives dequant 0.
// The search uses a reciprocal multiply for w'/step (its loss tolerance
// allows it); the pack reproduces the IEEE quotient exactly.
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
//
// fp64 arithmetic is slow on this part, and pow is the costliest of it.  A
// thread owns one channel j and up to kScaleCands candidates: log2(a_j)
// once, then per candidate y = exp2(alpha_k log2 a_j), both in fp64.  With the CUDA math
// library's documented maximum errors (1 ulp for log2 and for exp2) and
// |log2 a| <= 150 for any positive fp32 a, y is within (1.04 * 150 + 1) *
// 2^-52 relative of a^alpha, i.e. within 320 fp64 ulps.  Unless y lies within
// 2^10 ulps of a point where fp32 rounding changes (half-way between two fp32
// values), fp32(y) is fp32 of the exact power and of pow's result; near such
// a point the thread takes pow itself, so the table is what pow gives.
__device__ __forceinline__ float fp32_power(double a, double la, double alpha) {
  const double y = exp2(alpha * la);
  // bits below fp32 precision: 29 of the 52-bit fraction; the rounding point
  // is 1 followed by zeros there
  const long long bits = __double_as_longlong(y);
  const long long low = bits & ((1ll << 29) - 1);
  const long long dist = low >= (1ll << 28) ? low - (1ll << 28) : (1ll << 28) - low;
  const bool normal = y >= 1.1754943508222875e-38 && y <= 3.4028234663852886e38;  // fp32 normal range
  if (!normal || dist <= (1ll << 10)) return static_cast<float>(pow(a, alpha));
  return static_cast<float>(y);
}

constexpr int kScaleCands = 4;  // candidates per thread: blockIdx.y takes the next four

__global__ void scale_table_kernel(const float* __restrict__ mean_abs, int64_t D, AlphaGrid grid, int G,
                                   float act_floor, float* __restrict__ s_tab, float* __restrict__ r_tab,
                                   uint32_t* status) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= D) return;
  const float a = mean_abs[j];
  if (!isfinite(a) && blockIdx.y == 0) set_error(status, AWQ_DEV_NONFINITE);
  const double af = static_cast<double>(fmaxf(a, act_floor));
  const double la = log2(af);
  const int k1 = min(G, static_cast<int>(blockIdx.y + 1) * kScaleCands);
  for (int k = blockIdx.y * kScaleCands; k < k1; ++k) {
    const float s = isfinite(la) ? fp32_power(af, la, grid.a[k]) : static_cast<float>(pow(af, grid.a[k]));
    s_tab[static_cast<int64_t>(k) * D + j] = s;
    r_tab[static_cast<int64_t>(k) * D + j] = __fdiv_rn(1.0f, s);
  }
}

cudaError_t launch_scale_table(const float* mean_abs, int64_t D_in, const AlphaGrid& grid, int G, float act_floor,
                               float* s_tab, float* r_tab, uint32_t* status, cudaStream_t stream) {
  const dim3 g(static_cast<unsigned>((D_in + 127) / 128), static_cast<unsigned>((G + kScaleCands - 1) / kScaleCands));
  scale_table_kernel<<<g, 128, 0, stream>>>(mean_abs, D_in, grid, G, act_floor, s_tab, r_tab, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ group parameters
// Exact step / zero of one (group, column) from the range of its scaled weights.
// The closed-form scale of the aiqz.cc article (section 3):
//   s_i = (E|X_i|)^alpha / mean_j |W_ij|
// for input channel i (row i of W [D_in, D_out]).  One warp per row: 16-byte
// loads along the row, |w| accumulated in fp64 (a sum of bf16 magnitudes is
// exact in fp64 while the row spans at most ~30 binades, so the result does
// not depend on the order), a fixed-order warp tree; the quotient in fp64,
// rounded once to fp32.  The statistic is floored as for the grid search; a
// row of zeros gets s = 1.
__global__ void closed_form_kernel(const __nv_bfloat16* __restrict__ W, int64_t D_in, int64_t D_out,
                                   const float* __restrict__ mean_abs, double alpha, float act_floor,
                                   float* __restrict__ s_out) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= D_in) return;
  const __nv_bfloat16* wr = W + row * D_out;
  double acc = 0.0;
  for (int64_t c = static_cast<int64_t>(lane) * 8; c < D_out; c += 32 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(wr + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc += static_cast<double>(__uint_as_float((u[k] << 16) & 0x7FFFFFFFu));
      acc += static_cast<double>(__uint_as_float(u[k] & 0x7FFF0000u));
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) {
    const double den = acc / static_cast<double>(D_out);
    const double a = static_cast<double>(fmaxf(mean_abs[row], act_floor));
    s_out[row] = den > 0.0 ? static_cast<float>(pow(a, alpha) / den) : 1.f;
  }
}

cudaError_t launch_closed_form(const void* W, int64_t D_in, int64_t D_out, const float* mean_abs, double alpha,
                               float act_floor, float* s_out, cudaStream_t stream) {
  constexpr int kRowsPerCta = 8;
  closed_form_kernel<<<static_cast<unsigned>((D_in + kRowsPerCta - 1) / kRowsPerCta), kRowsPerCta * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(W), D_in, D_out, mean_abs, alpha, act_floor, s_out);
  return cudaGetLastError();
}

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
constexpr int kMaxGpCandidates = 21;  // candidates per CTA, the default grid (grid.z splits larger grids)
constexpr int kGpChunk = 64;          // rows of W staged per step (16 KB)

// The running range of one 64-row chunk for column t: for each quad of rows
// the thread unpacks its four weights once, then per candidate takes the
// quad's scales in one 16-byte broadcast load, forms w' = w s in two packed
// multiplies and folds them into the range with two three-input min / max
// operations.  FULL: all kMaxGpCandidates candidates are live (no per-candidate
// test in the loop).
template <bool FULL, bool SYM>
__device__ __forceinline__ void range_chunk(const __nv_bfloat16* wsh, const float4* ssh, int t, int nk,
                                            float (&lo)[kMaxGpCandidates], float (&hi)[kMaxGpCandidates]) {
  const uint16_t* wcol = reinterpret_cast<const uint16_t*>(wsh) + t;
#pragma unroll 1
  for (int rq = 0; rq < kGpChunk / 4; ++rq) {
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = __uint_as_float(static_cast<uint32_t>(wcol[(4 * rq + i) * kGpCols]) << 16);
    const float2 w01 = make_float2(w[0], w[1]), w23 = make_float2(w[2], w[3]);
    const float4* sp = ssh + rq * (FULL ? kMaxGpCandidates : nk);
#pragma unroll
    for (int k = 0; k < kMaxGpCandidates; ++k) {
      if (FULL || k < nk) {
        const float4 sq = sp[k];
        const float2 p = __fmul2_rn(w01, make_float2(sq.x, sq.y));
        const float2 q = __fmul2_rn(w23, make_float2(sq.z, sq.w));
        if (SYM) {
          hi[k] = fmaxabs3(fmaxabs3(hi[k], p.x, p.y), q.x, q.y);
        } else {
          lo[k] = fmin3(fmin3(lo[k], p.x, p.y), q.x, q.y);
          hi[k] = fmax3(fmax3(hi[k], p.x, p.y), q.x, q.y);
        }
      }
    }
  }
}

// One CTA: one group of GS rows x 128 columns, up to 21 candidates.  The group
// streams through shared memory in 64-row chunks (W chunk 16 KB, the chunk's
// scale rows as {s_k[r], .., s_k[r+3]} quads).  Thread t owns column t and
// keeps the running range of all candidates in registers (range_chunk).
// 22 KB of shared memory and <= 72 registers put 7 CTAs on an SM, so a
// 4096 x 4096 layer's 1024 CTAs run in one wave.
template <int GS>
__global__ void __launch_bounds__(kGpThreads, 6) group_params_kernel(const __nv_bfloat16* __restrict__ W,
                                                                const float* __restrict__ s_tab, int64_t D_in,
                                                                int64_t D_out, int G, int symmetric,
                                                                float* __restrict__ qp, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* wsh = reinterpret_cast<__nv_bfloat16*>(smem);            // [64][128]
  float4* ssh = reinterpret_cast<float4*>(smem + kGpChunk * kGpCols * 2);  // [16][nk]
  const int t = threadIdx.x;
  const int k0 = blockIdx.z * kMaxGpCandidates;
  const int nk = min(kMaxGpCandidates, G - k0);
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kGpCols;
  const int64_t grp = blockIdx.y;
  const int64_t n = n0 + t;
  bool bad = false;

  float lo[kMaxGpCandidates], hi[kMaxGpCandidates];
#pragma unroll
  for (int k = 0; k < kMaxGpCandidates; ++k) lo[k] = hi[k] = 0.f;

#pragma unroll 1
  for (int c0 = 0; c0 < GS; c0 += kGpChunk) {
    const int64_t j0 = grp * GS + c0;
    if (c0 > 0) __syncthreads();  // every thread is done with the previous chunk
    // the thread's W loads in two batches of four in flight (registers stay
    // below the bound that puts 7 CTAs on an SM)
    constexpr int kLoads = kGpChunk * (kGpCols / 8) / kGpThreads;
#pragma unroll
    for (int b = 0; b < kLoads; b += 4) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = t + (b + i) * kGpThreads;
        const int64_t col = n0 + (idx & 15) * 8;
        v[i] = col < D_out ? *reinterpret_cast<const uint4*>(W + (j0 + (idx >> 4)) * D_out + col)
                           : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = t + (b + i) * kGpThreads;
        bad |= bf16x2_nonfinite(v[i].x) | bf16x2_nonfinite(v[i].y) | bf16x2_nonfinite(v[i].z) |
               bf16x2_nonfinite(v[i].w);
        *reinterpret_cast<uint4*>(wsh + (idx >> 4) * kGpCols + (idx & 15) * 8) = v[i];
      }
    }
    {
      // scale quads of the chunk, up to kMaxGpCandidates * 16 of them (rounded
      // up to whole rounds of the CTA; the k < nk test skips the overhang)
      constexpr int kSLoads = (kMaxGpCandidates * (kGpChunk / 4) + kGpThreads - 1) / kGpThreads;
      float4 sv[kSLoads];
#pragma unroll
      for (int i = 0; i < kSLoads; ++i) {
        const int idx = t + i * kGpThreads;
        const int k = idx / (kGpChunk / 4);
        const int rq = idx - k * (kGpChunk / 4);
        sv[i] = k < nk ? *reinterpret_cast<const float4*>(s_tab + static_cast<int64_t>(k0 + k) * D_in + j0 + 4 * rq)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < kSLoads; ++i) {
        const int idx = t + i * kGpThreads;
        const int k = idx / (kGpChunk / 4);
        const int rq = idx - k * (kGpChunk / 4);
        if (k < nk) ssh[rq * nk + k] = sv[i];
      }
    }
    __syncthreads();
    if (n < D_out) {
      if (nk == kMaxGpCandidates) {
        if (symmetric)
          range_chunk<true, true>(wsh, ssh, t, nk, lo, hi);
        else
          range_chunk<true, false>(wsh, ssh, t, nk, lo, hi);
      } else {
        if (symmetric)
          range_chunk<false, true>(wsh, ssh, t, nk, lo, hi);
        else
          range_chunk<false, false>(wsh, ssh, t, nk, lo, hi);
      }
    }
  }
  if (bad && blockIdx.z == 0) set_error(status, AWQ_DEV_NONFINITE);
  // every thread of the warp takes part in the chunk flags' ballot below
  const bool valid = n < D_out;
  const int64_t T = D_in / GS;
  const int64_t kstride = T * (D_out / kQChunkCols) * kQChunkFloats;
  float* dst0 = qp + k0 * kstride + (grp * (D_out / kQChunkCols) + n / kQChunkCols) * kQChunkFloats +
                (n % kQChunkCols);
  const int lane = t & 31;
  // the code range with the table's offset: zm = 1.5*2^23 + zero, and zero 0
  // for symmetric codes (stored +8 only by the pack)
  const float qlo = symmetric ? kMagic - 7.f : kMagic, qhi = symmetric ? kMagic + 7.f : kMagic + 15.f;
#pragma unroll
  for (int k = 0; k < kMaxGpCandidates; ++k) {
    if (k < nk) {
      const QParam q = make_qparam(lo[k], hi[k], symmetric, status);
      // The codes of a column leave the code range only at its extremes:
      // rint is monotone, so the column's largest code is the one of the
      // range's top, fma(hi, 1/step, 1.5*2^23 + zero), and its smallest the
      // one of the range's bottom, formed with the same fused multiply-add
      // and rounding as the searches' and the pack's codes.  A non-finite
      // range fails both comparisons.
      const float bottom = symmetric ? -hi[k] : lo[k];
      const bool need = valid && !(__fmaf_rn(hi[k], q.inv, q.zm) <= qhi && __fmaf_rn(bottom, q.inv, q.zm) >= qlo);
      const uint32_t chunk_bits = (__ballot_sync(0xFFFFFFFFu, need) >> (lane & ~(kQChunkCols - 1))) & 0xFFu;
      if (valid) {
        float* dst = dst0 + k * kstride;
        dst[0] = q.inv;
        dst[kQChunkCols] = q.zm;
        dst[2 * kQChunkCols] = q.step;
        if ((n % kQChunkCols) == 0) dst[3 * kQChunkCols] = chunk_bits ? 1.f : 0.f;
      }
    }
  }
}

static size_t group_params_smem(int) {
  return static_cast<size_t>(kGpChunk) * kGpCols * 2 + static_cast<size_t>(kGpChunk / 4) * kMaxGpCandidates * 16;
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

}  // namespace awqdev
