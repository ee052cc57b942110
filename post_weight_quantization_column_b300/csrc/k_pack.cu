// Step 4: offline quantisation and nibble packing of diag(s) W.
// "AWQ (Activation-aware Weight Quantization)", 推理时的等效实现:
// W_quantized = Quantize(diag(s*) W); "009. AWQ Integration", Consequences:
// two 4-bit codes per byte (even input row in the low nibble).
//
// Quantiser (技术原理 - 量化数学基础; aiqz.cc article
// "awq-activation-aware-quantization", section 4; the asymmetric zero-point
// form of the CSDN AutoAWQ walkthrough's quant_config):
//   asymmetric: step = fp16((max(w',0) - min(w',0)) / 15), zero = clamp(rint(-min/step), 0, 15),
//               code = clamp(rint(w'/step) + zero, 0, 15)
//   symmetric:  step = fp16(max|w'| / 7), code = clamp(rint(w'/step), -7, 7) + 8, zero 8
//
// Two HBM-bound streaming kernels, both one pass over W with a thread's
// 8 rows x 8 columns (one 16-byte load per row) held in registers:
//   pack_kernel           any s (awq_quantize_pack): the CTA also forms the
//                         per-column range of its group(s) and the exact
//                         step / zero before it emits the codes;
//   pack_searched_kernel  right after a search, whose parameter table already
//                         holds the step / zero of every (group, column) for
//                         the best candidate.
//
// Codes equal clamp(rint(fp32(w'/step)) + zero): the quotient is first
// formed as w' * (1/step); where that lands within 8e-6 of a half-integer
// (where the two could round differently), the thread redoes its rows with
// the IEEE division.  |w'/step| <= 45 in every case, where the product is
// within 6e-6 of the IEEE quotient, so elsewhere both round alike.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {
namespace {

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kTieGuard = 0.5f - 8.0e-6f;
constexpr int kPackRows = 8;       // rows per thread: four row pairs, one packed byte row each
constexpr int kPackThreads = 256;  // both kernels

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
// The same two values by byte permutes: the range pass unpacks with these and
// the code pass with the shifts above, so that the compiler recomputes them
// instead of keeping 64 unpacked floats live across the barrier.
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  return make_float2(__uint_as_float(__byte_perm(u, 0u, 0x1044)), __uint_as_float(__byte_perm(u, 0u, 0x3244)));
}
// Running range helpers.  The .NaN forms propagate a NaN operand, so a
// non-finite weight (or scale) leaves a non-finite range behind, which the
// step / zero phase reports; on finite inputs they are exact min / max.
__device__ __forceinline__ float nmin3(float a, float b, float c) {
  float d;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float nmax3(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float nmaxabs3(float a, float b, float c) {  // max(|a|, |b|, |c|)
  float d;
  asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float nmin(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float nmax(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float maxabs3(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Codes of one thread's 8 rows x 8 columns through the reciprocal.  For each
// weight c = fma(w', 1/step, 1.5*2^23 + zero) rounds the exact product to an
// integer code; d = rint - w'/step (one more fma) is within 1/2 of it, and
// the returned maximum |d| flags a near tie anywhere in the thread's
// elements.  Each packed byte is c_even + 16 c_odd in the low bits
// (1.5*2^23 has a zero low byte).  Asymmetric codes get no lower clamp here:
// rint is odd, so while the zero equals rint(-min/step) the group minimum
// gets code 0 and every other element more.  That fails only where the zero
// was clamped to 15 (a subnormal fp16 step that rounded far down can put
// -min/step above 15.5), so callers send every thread with a zero of 15 in
// its columns to the exact path (see has_zero15).
// inv, zmz: 1/step and 1.5*2^23 + the stored offset (the zero; 8 for
// symmetric codes) of the 8 columns; out[p]: the 8 bytes of row pair p.
// CLAMP = false drops the upper clamp (and the symmetric lower one) for
// columns whose largest code is known to stay in range.
template <bool SYM, bool CLAMP = true>
__device__ __forceinline__ float codes_8x8(const uint4 (&w)[kPackRows], const float (&sj)[kPackRows],
                                           const float (&inv)[8], const float (&zmz)[8],
                                           uint32_t (&out)[kPackRows / 2][2]) {
  const float clo = SYM ? kMagic + 1.f : kMagic;
  const float chi = kMagic + 15.f;
  float tmax = 0.f;
#pragma unroll
  for (int p = 0; p < kPackRows / 2; ++p) {
    const uint32_t we[4] = {w[2 * p].x, w[2 * p].y, w[2 * p].z, w[2 * p].w};
    const uint32_t wo[4] = {w[2 * p + 1].x, w[2 * p + 1].y, w[2 * p + 1].z, w[2 * p + 1].w};
    uint32_t half16[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 inv2 = make_float2(inv[2 * j], inv[2 * j + 1]);
      const float2 ninv2 = make_float2(-inv[2 * j], -inv[2 * j + 1]);
      const float2 zm2 = make_float2(zmz[2 * j], zmz[2 * j + 1]);
      const float2 nzm2 = make_float2(-zmz[2 * j], -zmz[2 * j + 1]);
      const float2 pe = __fmul2_rn(make_float2(bf16lo(we[j]), bf16hi(we[j])), make_float2(sj[2 * p], sj[2 * p]));
      const float2 po =
          __fmul2_rn(make_float2(bf16lo(wo[j]), bf16hi(wo[j])), make_float2(sj[2 * p + 1], sj[2 * p + 1]));
      float2 ce = __ffma2_rn(pe, inv2, zm2);
      float2 co = __ffma2_rn(po, inv2, zm2);
      const float2 de = __ffma2_rn(pe, ninv2, __fadd2_rn(ce, nzm2));
      const float2 dd = __ffma2_rn(po, ninv2, __fadd2_rn(co, nzm2));
      tmax = maxabs3(tmax, de.x, de.y);
      tmax = maxabs3(tmax, dd.x, dd.y);
      if (SYM && CLAMP) {
        ce.x = fmaxf(ce.x, clo);
        ce.y = fmaxf(ce.y, clo);
        co.x = fmaxf(co.x, clo);
        co.y = fmaxf(co.y, clo);
      }
      if (CLAMP) {
        ce.x = fminf(ce.x, chi);
        ce.y = fminf(ce.y, chi);
        co.x = fminf(co.x, chi);
        co.y = fminf(co.y, chi);
      }
      const uint32_t x0 = __float_as_uint(co.x) * 16u + __float_as_uint(ce.x);  // byte 2j in the low 8 bits
      const uint32_t x1 = __float_as_uint(co.y) * 16u + __float_as_uint(ce.y);  // byte 2j+1
      half16[j] = __byte_perm(x0, x1, 0x0040);
    }
    out[p][0] = __byte_perm(half16[0], half16[1], 0x5410);
    out[p][1] = __byte_perm(half16[2], half16[3], 0x5410);
  }
  return tmax;
}

// The exact path of one thread's 8 rows x 8 columns (rare: only where some
// quotient lies within the tie guard of a half step): codes from the IEEE
// fp32 quotient w'/step, as the oracle defines them, written to qweight.
// qc: {1/step x8, 1.5*2^23 + zero x8, step x8} of the thread's 8 columns (in
// the search's parameter table or in shared memory).  Kept out of line so
// that its registers do not burden the streaming path.
template <bool SYM>
__device__ __noinline__ void pack_exact_8x8(const __nv_bfloat16* __restrict__ W, const float* __restrict__ s,
                                            const float* __restrict__ qc, int64_t row0, int64_t n, int64_t D_out,
                                            uint8_t* __restrict__ qweight) {
  for (int p = 0; p < kPackRows / 2; ++p) {
    const uint4 a = *reinterpret_cast<const uint4*>(W + (row0 + 2 * p) * D_out + n);
    const uint4 b = *reinterpret_cast<const uint4*>(W + (row0 + 2 * p + 1) * D_out + n);
    const float se = s[row0 + 2 * p], so = s[row0 + 2 * p + 1];
    const uint32_t we[4] = {a.x, a.y, a.z, a.w};
    const uint32_t wo[4] = {b.x, b.y, b.z, b.w};
    uint32_t bytes[8];
    for (int j = 0; j < 8; ++j) {
      const float xe = (j & 1) ? bf16hi(we[j >> 1]) : bf16lo(we[j >> 1]);
      const float xo = (j & 1) ? bf16hi(wo[j >> 1]) : bf16lo(wo[j >> 1]);
      const float step = qc[2 * kQChunkCols + j];
      const float zo = SYM ? 8.f : qc[kQChunkCols + j] - kMagic;
      const float ql = SYM ? 1.f : 0.f;
      // clamp(rint(IEEE w'/step) + zero, ql, 15); a zero step keeps the zero
      uint32_t ke = static_cast<uint32_t>(zo), ko = ke;
      if (step != 0.f) {
        const float qe = rintf(__fdiv_rn(__fmul_rn(xe, se), step)) + zo;
        const float qo = rintf(__fdiv_rn(__fmul_rn(xo, so), step)) + zo;
        ke = static_cast<uint32_t>(fminf(fmaxf(qe, ql), 15.f));
        ko = static_cast<uint32_t>(fminf(fmaxf(qo, ql), 15.f));
      }
      bytes[j] = ke | (ko << 4);
    }
    *reinterpret_cast<uint2*>(qweight + (row0 / 2 + p) * D_out + n) =
        make_uint2(bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24),
                   bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24));
  }
}

// An asymmetric zero of 15 in any of the thread's columns: the codes need
// the lower clamp of the exact path (rare: one-signed negative groups).
template <bool SYM>
__device__ __forceinline__ bool has_zero15(const float (&zmz)[8]) {
  if (SYM) return false;
  bool z15 = false;
#pragma unroll
  for (int k = 0; k < 8; ++k) z15 |= zmz[k] == kMagic + 15.f;
  return z15;
}

__device__ __forceinline__ void store_codes_8x8(const uint32_t (&out)[kPackRows / 2][2], int64_t row0, int64_t n,
                                                int64_t D_out, uint8_t* __restrict__ qweight) {
#pragma unroll
  for (int p = 0; p < kPackRows / 2; ++p)
    *reinterpret_cast<uint2*>(qweight + (row0 / 2 + p) * D_out + n) = make_uint2(out[p][0], out[p][1]);
}

// ---------------------------------------------------------------------------
// Pack at any s.  A CTA of 256 threads holds ROWS rows (one group of 128 or
// 256, two groups of 64) x COLS columns of W in registers: thread = one row
// block of 8 rows x one chunk of 8 columns, the CW chunks of a row block on
// consecutive lanes, so that a warp reads CW * 16 contiguous bytes of each
// of its rows.  The per-column range of w' = w * s is combined over the row
// blocks of a warp by shuffles, then over the warps of a group in shared
// memory (min / max are exact, so the order does not matter); one thread per
// (group, column) forms the exact step and zero, writes the fp16 scale and
// zero, and leaves {1/step, 1.5*2^23 + zero, step} in shared memory, from
// which every thread emits its codes.
template <int GS>
struct PackShape {
  static constexpr int CW = GS == 256 ? 8 : 16;  // chunks of 8 columns per CTA
  static constexpr int RBW = 32 / CW;            // row blocks per warp
  static constexpr int WARPS = kPackThreads / 32;
  static constexpr int ROWS = WARPS * RBW * kPackRows;  // 128 or 256
  static constexpr int GROUPS = ROWS / GS;              // groups per CTA
  static constexpr int WPG = WARPS / GROUPS;            // warps per group
  static constexpr int COLS = CW * kQChunkCols;         // 128 or 64
  static_assert(GROUPS >= 1 && WPG * GROUPS == WARPS, "a group is whole warps");
};
constexpr int kRangePad = 12;  // floats per chunk in the range exchange: 8 chunks of a quarter-warp on disjoint banks

template <int GS, bool SYM>
__global__ void __launch_bounds__(kPackThreads, 3)
    pack_kernel(const __nv_bfloat16* __restrict__ W, const float* __restrict__ s, int64_t D_in, int64_t D_out,
                uint8_t* __restrict__ qweight, __half* __restrict__ scales, __half* __restrict__ zeros,
                uint32_t* status) {
  using P = PackShape<GS>;
  __shared__ __align__(16) float red_lo[SYM ? 1 : P::WARPS][P::CW * kRangePad];
  __shared__ __align__(16) float red_hi[P::WARPS][P::CW * kRangePad];
  __shared__ __align__(16) float prm[P::GROUPS][P::CW * kQChunkFloats];  // the search table's chunk layout
  __shared__ __align__(8) uint8_t clampc[P::GROUPS][P::COLS];  // 1: the column's codes need the clamps

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int c = lane % P::CW;
  const int rb = warp * P::RBW + lane / P::CW;  // row block in the CTA
  const int gi = warp / P::WPG;                 // group in the CTA
  const int64_t n = static_cast<int64_t>(blockIdx.x) * P::COLS + c * kQChunkCols;
  const int64_t row0 = static_cast<int64_t>(blockIdx.y) * P::ROWS + rb * kPackRows;
  const bool rows_ok = row0 < D_in;  // D_in is a multiple of GS: a group lies wholly inside or outside
  const bool active = rows_ok && n < D_out;

  uint4 w[kPackRows];
  float sj[kPackRows];
#pragma unroll
  for (int i = 0; i < kPackRows; ++i) {
    w[i] = active ? *reinterpret_cast<const uint4*>(W + (row0 + i) * D_out + n) : make_uint4(0u, 0u, 0u, 0u);
    sj[i] = rows_ok ? s[row0 + i] : 0.f;
  }

  // range of w' over the thread's rows (zeros included; NaN-propagating),
  // then over the row blocks of the warp: lanes c, c + CW, ...
  float lo[8], hi[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) lo[k] = hi[k] = 0.f;
#pragma unroll
  for (int r = 0; r < kPackRows; r += 2) {
    const uint32_t we[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
    const uint32_t wo[4] = {w[r + 1].x, w[r + 1].y, w[r + 1].z, w[r + 1].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 pe = __fmul2_rn(unpack_bf16x2(we[k]), make_float2(sj[r], sj[r]));
      const float2 po = __fmul2_rn(unpack_bf16x2(wo[k]), make_float2(sj[r + 1], sj[r + 1]));
      if (SYM) {
        hi[2 * k] = nmaxabs3(hi[2 * k], pe.x, po.x);
        hi[2 * k + 1] = nmaxabs3(hi[2 * k + 1], pe.y, po.y);
      } else {
        lo[2 * k] = nmin3(lo[2 * k], pe.x, po.x);
        hi[2 * k] = nmax3(hi[2 * k], pe.x, po.x);
        lo[2 * k + 1] = nmin3(lo[2 * k + 1], pe.y, po.y);
        hi[2 * k + 1] = nmax3(hi[2 * k + 1], pe.y, po.y);
      }
    }
  }
#pragma unroll
  for (int off = P::CW; off < 32; off <<= 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (!SYM) lo[k] = nmin(lo[k], __shfl_xor_sync(0xFFFFFFFFu, lo[k], off));
      hi[k] = nmax(hi[k], __shfl_xor_sync(0xFFFFFFFFu, hi[k], off));
    }
  }
  if (lane < P::CW) {
    float4* dh = reinterpret_cast<float4*>(&red_hi[warp][c * kRangePad]);
    dh[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
    dh[1] = make_float4(hi[4], hi[5], hi[6], hi[7]);
    if (!SYM) {
      float4* dl = reinterpret_cast<float4*>(&red_lo[warp][c * kRangePad]);
      dl[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
      dl[1] = make_float4(lo[4], lo[5], lo[6], lo[7]);
    }
  }
  __syncthreads();

  if (t < P::GROUPS * P::COLS) {
    // exact step / zero of one (group, column)
    const int g2 = t / P::COLS, col = t % P::COLS;
    const int pc = (col >> 3) * kRangePad + (col & 7);
    float l = 0.f, h = 0.f;
#pragma unroll
    for (int k = 0; k < P::WPG; ++k) {
      if (!SYM) l = nmin(l, red_lo[g2 * P::WPG + k][pc]);
      h = nmax(h, red_hi[g2 * P::WPG + k][pc]);
    }
    const int64_t ncol = static_cast<int64_t>(blockIdx.x) * P::COLS + col;
    const int64_t grp = static_cast<int64_t>(blockIdx.y) * P::GROUPS + g2;
    const bool valid = ncol < D_out && grp * GS < D_in;
    float sc = 0.f;
    if (!isfinite(l) || !isfinite(h)) {
      if (valid) set_error(status, AWQ_DEV_NONFINITE);  // codes of this column stay at the zero
    } else {
      const float raw = SYM ? __fdiv_rn(h, 7.0f) : __fdiv_rn(__fsub_rn(h, l), 15.0f);
      sc = __half2float(__float2half_rn(raw));
      if (isinf(sc)) {
        if (valid) set_error(status, AWQ_DEV_RANGE);
        sc = 0.f;
      }
    }
    float z = 0.f;
    // an integer code in [0, 15]; the int round trip also turns -0 into +0
    if (!SYM && sc != 0.f) z = static_cast<float>(static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(-l, sc)), 0.f), 15.f)));
    // Every element lies in [l, h], and rint is monotone, so outside near
    // ties (the exact path) the largest code is rint(h/step) + zero
    // (asymmetric) or rint(max|w'|/step) + 8 with max|w'| < 7.5 step
    // (symmetric; 7.5 step is exact for an fp16 step).  Columns where that
    // can leave the code range, and non-finite ones, keep the clamps.
    bool need = !isfinite(l) || !isfinite(h);
    if (sc != 0.f) need = need || (SYM ? h >= 7.5f * sc : rintf(__fdiv_rn(h, sc)) + z > 15.f);
    clampc[g2][col] = need ? 1 : 0;
    float* q = &prm[g2][(col >> 3) * kQChunkFloats + (col & 7)];
    q[0] = sc != 0.f ? __frcp_rn(sc) : 0.f;
    q[kQChunkCols] = kMagic + (SYM ? 8.f : z);
    q[2 * kQChunkCols] = sc;
    if (valid) {
      scales[grp * D_out + ncol] = __float2half_rn(sc);
      zeros[grp * D_out + ncol] = __float2half_rn(SYM ? 8.f : z);
    }
  }
  __syncthreads();
  if (!active) return;

  const float* qc = &prm[gi][c * kQChunkFloats];
  float inv[8], zmz[8];
  {
    const float4* q4 = reinterpret_cast<const float4*>(qc);
    const float4 i0 = q4[0], i1 = q4[1], z0 = q4[2], z1 = q4[3];
    const float ia[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
    const float za[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      inv[k] = ia[k];
      zmz[k] = za[k];
    }
  }
  uint32_t out[kPackRows / 2][2];
  const uint2 cf = *reinterpret_cast<const uint2*>(&clampc[gi][c * kQChunkCols]);
  const bool clampw = __any_sync(__activemask(), (cf.x | cf.y) != 0u);  // one path per warp
  const float tmax = clampw ? codes_8x8<SYM, true>(w, sj, inv, zmz, out) : codes_8x8<SYM, false>(w, sj, inv, zmz, out);
  if (tmax > kTieGuard || has_zero15<SYM>(zmz)) {
    pack_exact_8x8<SYM>(W, s, qc, row0, n, D_out, qweight);
    return;
  }
  store_codes_8x8(out, row0, n, D_out, qweight);
}

template <int GS, bool SYM>
cudaError_t launch_pack_t(const void* W, const float* s, int64_t D_in, int64_t D_out, uint8_t* qweight,
                          void* scales, void* zeros, uint32_t* status, cudaStream_t stream) {
  using P = PackShape<GS>;
  const dim3 grid(static_cast<unsigned>((D_out + P::COLS - 1) / P::COLS),
                  static_cast<unsigned>((D_in + P::ROWS - 1) / P::ROWS));
  pack_kernel<GS, SYM><<<grid, kPackThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(W), s, D_in, D_out,
                                                          qweight, static_cast<__half*>(scales),
                                                          static_cast<__half*>(zeros), status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Pack after a search.  The search's group-parameter pass already holds, for
// every candidate, the exact step (fp16-rounded range / 15 or max|w'| / 7),
// 1/step, zero and clamp flag of every (group, column) -- the same formulas
// and the same exact ranges as pack_kernel forms.  For its best candidate the
// pack is then a single streaming pass with no exchange between threads: a
// thread owns 8 columns (chunk c) x 8 rows (row block rb) of one group, loads
// all 8 rows at once and emits codes as pack_kernel does; the threads of row
// block 0 of a group write its fp16 scales and zeros.  Grid: x = blocks of
// 256 chunks (a warp reads 512 contiguous bytes of a row), y = row blocks
// (strided over when there are more than the grid's y extent), so a thread
// finds its place without divisions.
template <int GS, bool SYM>
__global__ void __launch_bounds__(kPackThreads, 3)
    pack_searched_kernel(const __nv_bfloat16* __restrict__ W, const float* __restrict__ s,
                         const float* __restrict__ qp, const int32_t* __restrict__ best_idx, int G, int64_t D_in,
                         int64_t D_out, uint8_t* __restrict__ qweight, __half* __restrict__ scales,
                         __half* __restrict__ zeros) {
  const int64_t chunks = D_out / kQChunkCols;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kPackThreads + threadIdx.x;
  if (c >= chunks) return;
  const int64_t T = D_in / GS;
  const int64_t n = c * kQChunkCols;
  int k = *best_idx;
  k = k < 0 ? 0 : (k >= G ? G - 1 : k);  // awq_search always writes an index in [0, G)
  for (int64_t rbg = blockIdx.y; rbg < D_in / kPackRows; rbg += gridDim.y) {
  const int64_t row0 = rbg * kPackRows;
  const int64_t g = row0 / GS;
  const bool first_block = (row0 % GS) == 0;

  uint4 w[kPackRows];
#pragma unroll
  for (int i = 0; i < kPackRows; ++i) w[i] = *reinterpret_cast<const uint4*>(W + (row0 + i) * D_out + n);
  float sj[kPackRows];
#pragma unroll
  for (int i = 0; i < kPackRows; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(s + row0 + i);  // s_star: 16-byte aligned (checked)
    sj[i] = v.x;
    sj[i + 1] = v.y;
    sj[i + 2] = v.z;
    sj[i + 3] = v.w;
  }
  // {1/step x8, 1.5*2^23 + zero x8, step x8, clamp flag, ...} of (best candidate, group, chunk)
  const float* qc = qp + ((static_cast<int64_t>(k) * T + g) * chunks + c) * kQChunkFloats;
  const float4* q4 = reinterpret_cast<const float4*>(qc);
  float inv[8], zmz[8];  // zmz: 1.5*2^23 + the stored offset (the zero; 8 for symmetric codes)
  {
    const float4 i0 = q4[0], i1 = q4[1];
    const float ia[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) inv[j] = ia[j];
    if (SYM) {
#pragma unroll
      for (int j = 0; j < 8; ++j) zmz[j] = kMagic + 8.f;
    } else {
      const float4 z0 = q4[2], z1 = q4[3];
      const float za[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) zmz[j] = za[j];
    }
  }
  if (first_block) {
    const float4 s0 = q4[4], s1 = q4[5];
    const float st[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t sc[4], zr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 hs = __floats2half2_rn(st[2 * j], st[2 * j + 1]);
      const __half2 hz = __floats2half2_rn(zmz[2 * j] - kMagic, zmz[2 * j + 1] - kMagic);
      sc[j] = *reinterpret_cast<const uint32_t*>(&hs);
      zr[j] = *reinterpret_cast<const uint32_t*>(&hz);
    }
    *reinterpret_cast<uint4*>(scales + g * D_out + n) = make_uint4(sc[0], sc[1], sc[2], sc[3]);
    *reinterpret_cast<uint4*>(zeros + g * D_out + n) = make_uint4(zr[0], zr[1], zr[2], zr[3]);
  }
  uint32_t out[kPackRows / 2][2];
  // the table's clamp flag, for the same codes the search formed; one path per warp
  const bool clampw = __any_sync(__activemask(), qc[kQChunkClamp] != 0.f);
  const float tmax = clampw ? codes_8x8<SYM, true>(w, sj, inv, zmz, out) : codes_8x8<SYM, false>(w, sj, inv, zmz, out);
  if (tmax > kTieGuard || has_zero15<SYM>(zmz)) {
    pack_exact_8x8<SYM>(W, s, qc, row0, n, D_out, qweight);
  } else {
    store_codes_8x8(out, row0, n, D_out, qweight);
  }
  }
}

template <int GS, bool SYM>
cudaError_t launch_pack_searched_t(const void* W, const float* s, const float* qp, const int32_t* best_idx, int G,
                                   int64_t D_in, int64_t D_out, uint8_t* qweight, void* scales, void* zeros,
                                   cudaStream_t stream) {
  const int64_t xblocks = (D_out / kQChunkCols + kPackThreads - 1) / kPackThreads;
  const int64_t yblocks = std::min<int64_t>(D_in / kPackRows, 65535);
  const dim3 grid(static_cast<unsigned>(xblocks), static_cast<unsigned>(yblocks));
  pack_searched_kernel<GS, SYM><<<grid, kPackThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(W), s, qp, best_idx, G, D_in, D_out, qweight, static_cast<__half*>(scales),
      static_cast<__half*>(zeros));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(const void* W, const float* s, int64_t D_in, int64_t D_out, int group_size, int symmetric,
                        uint8_t* qweight, void* scales, void* zeros, uint32_t* status, cudaStream_t stream) {
#define AWQ_PACK(GS)                                                                                              \
  return symmetric ? launch_pack_t<GS, true>(W, s, D_in, D_out, qweight, scales, zeros, status, stream)          \
                   : launch_pack_t<GS, false>(W, s, D_in, D_out, qweight, scales, zeros, status, stream)
  switch (group_size) {
    case 64:
      AWQ_PACK(64);
    case 128:
      AWQ_PACK(128);
    case 256:
      AWQ_PACK(256);
    default:
      return cudaErrorInvalidValue;
  }
#undef AWQ_PACK
}

cudaError_t launch_pack_searched(const void* W, const float* s, const float* qp, const int32_t* best_idx, int G,
                                 int64_t D_in, int64_t D_out, int group_size, int symmetric, uint8_t* qweight,
                                 void* scales, void* zeros, cudaStream_t stream) {
#define AWQ_PACK_SEARCHED(GS)                                                                                      \
  return symmetric ? launch_pack_searched_t<GS, true>(W, s, qp, best_idx, G, D_in, D_out, qweight, scales, zeros,   \
                                                      stream)                                                     \
                   : launch_pack_searched_t<GS, false>(W, s, qp, best_idx, G, D_in, D_out, qweight, scales, zeros, \
                                                       stream)
  switch (group_size) {
    case 64:
      AWQ_PACK_SEARCHED(64);
    case 128:
      AWQ_PACK_SEARCHED(128);
    case 256:
      AWQ_PACK_SEARCHED(256);
    default:
      return cudaErrorInvalidValue;
  }
#undef AWQ_PACK_SEARCHED
}

}  // namespace awqdev
