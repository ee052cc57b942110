// The ADR's second search: per-group coordinate greedy over power-of-two
// channel scales ("009. AWQ Integration", 关键设计 1-3).  Groups of g input
// rows are independent; inside a group, channel j in turn tries every
// candidate 2^k, the group's activation-weighted reconstruction error
//   E_group = sum_i a_i sum_n (w'hat_in / s_i - w_in)^2,  w' = w s,
// is evaluated with the pack's own quantiser for each, and the best is kept
// (a candidate replaces the current scale only when strictly better; the
// first in k order among equals).  Several passes over the group.
//
// One launch per channel position j of every group (all groups at once):
// grid (column slices of 128, groups), one column per thread.  A thread
// forms its column's range without channel j, the error of the other rows
// under the step / zero of that range, and then for each candidate only
// the term of channel j -- unless the scaled channel widens the range, in
// which case it re-sums the column under the new step / zero.  The group's
// rows sit in shared memory as row pairs (two bf16 of one column in a
// word), so that packed fp32 operations take two rows at once, and each
// row's term is taken in the scaled space: with s a power of two,
//   a (w'hat / s - w)^2 = (a / s^2) (w'hat - w')^2
// exactly, so a row needs only s and a / s^2.  Codes are rint of the IEEE
// quotient w'/step as the oracle defines them, formed as w' * (1/step) and
// redone with the division within 8e-6 of a half step (w s and step / s are
// exact).  Column errors are summed in a fixed order (two interleaved
// partial sums over the row pairs, a warp tree per candidate, then the
// warps in order), the slices of a group in slice order in fp64 by the last
// CTA of the group to finish (ticket counter), which also takes the
// decision and updates the scale.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {
namespace {

constexpr int kGreedyCols = 128;  // columns per CTA (one per thread)

struct Range {
  float lo, hi;  // asymmetric: min / max of w' with 0 included; symmetric: hi = max |w'|
};

struct Quant {
  float step, zero;  // zero: the asymmetric zero point (0 for symmetric codes)
  float inv;         // RN(1 / step) (0 for a zero step)
  // the codes of the range's own elements can leave the code range: an
  // asymmetric zero clamped at 15 (rint(-lo/step) > 15) or a symmetric
  // max|w'| >= 7.5 step -- both only where a subnormal fp16 step rounded far
  // down; the column sums then take the clamped exact form
  bool wide;
};

// Within this distance of a half step the reciprocal product and the IEEE
// quotient can round differently: |w'/step| <= 45 in every case, where the
// product is within 6e-6 of the quotient.
constexpr float kTieGuard = 0.5f - 8.0e-6f;

template <bool SYM>
__device__ __forceinline__ Quant quant_of(Range r, uint32_t* status) {
  Quant q;
  const float raw = SYM ? __fdiv_rn(r.hi, 7.0f) : __fdiv_rn(__fsub_rn(r.hi, r.lo), 15.0f);
  float sc = __half2float(__float2half_rn(raw));
  if (isinf(sc)) {
    set_error(status, AWQ_DEV_RANGE);
    sc = 0.f;
  }
  q.step = sc;
  const float zr = (!SYM && sc != 0.f) ? rintf(__fdiv_rn(-r.lo, sc)) : 0.f;
  q.zero = fminf(fmaxf(zr, 0.f), 15.f);
  q.inv = sc != 0.f ? __frcp_rn(sc) : 0.f;
  q.wide = SYM ? (sc != 0.f && r.hi >= 7.5f * sc) : zr > 15.f;  // 7.5 sc is exact (sc is an fp16 value)
  return q;
}

// a * (w'hat / s - w)^2 for one weight w with scale s and rs = 1/s (powers of
// two), with both clamps: the term of channel j under a candidate scale.
// The fast form takes rint(w' * (1/step)) and raises `dev` to the distance
// of that product from its rounding; where dev ends above the tie guard the
// caller redoes the term with the exact form (rint of the IEEE quotient).
template <bool SYM, bool EXACT>
__device__ __forceinline__ float term(float w, float s, float rs, float a, Quant q, float& dev) {
  float d;
  if (q.step == 0.f) {
    d = -w;
  } else {
    const float wp = w * s;  // exact
    float t;
    if (EXACT) {
      t = rintf(__fdiv_rn(wp, q.step));
    } else {
      const float tq = wp * q.inv;
      t = rintf(tq);
      dev = fmaxf(dev, fabsf(tq - t));
    }
    const float c = SYM ? fminf(fmaxf(t, -7.f), 7.f) : fminf(fmaxf(t + q.zero, 0.f), 15.f) - q.zero;
    d = fmaf(c, q.step * rs, -w);  // (code - zero) * step / s exact; one rounding of the difference
  }
  return a * (d * d);
}

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: x + kMagic rounds x to an integer (|x| < 2^22)

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
// three-input min / max (a NaN operand is ignored, as by fminf / fmaxf)
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float maxabs3f(float a, float b, float c) {  // max(|a|, |b|, |c|)
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// sum over the group's rows of one column: row pair p of column t is
// wt2[p][t] (row 2p in the low half), rowc[p] = {s_2p, s_2p+1, b_2p, b_2p+1}
// with b = a / s^2 (0 for channel jj, whose weight is also zeroed).
// The fast form takes r = rint(w' * (1/step)) through the 1.5*2^23 sum, and
// the largest |r - w'/step| over the rows flags a near tie; there, and where
// q.wide is set, the column is redone with the clamped IEEE quotient.
// Otherwise codes need no clamp below (asymmetric: rint is odd, so with the
// zero equal to rint(-lo/step) the group minimum gets code 0 and the rest
// more; symmetric: max|w'| < 7.5 step puts rint(w'/step) in [-7, 7]), and
// above only for asymmetric codes, where the fp16 rounding of the step can
// give 16.
template <int GS, bool SYM>
__device__ __forceinline__ float column_error(const uint32_t (*wt2)[kGreedyCols], const float4* rowc, int t, Quant q) {
  const float2 inv2 = make_float2(q.inv, q.inv), ninv2 = make_float2(-q.inv, -q.inv);
  const float zm = kMagic + q.zero;
  const float2 zm2 = make_float2(zm, zm), nzm2 = make_float2(-zm, -zm);
  const float2 nstep2 = make_float2(-q.step, -q.step);
  const float hic = 15.f - q.zero;
  float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
  float dev = q.wide ? 1.f : 0.f;  // 1: straight to the exact form
  // (r step - w')^2 = (w' - r step)^2: the negated difference is one fma;
  // a zero step (inv 0, r 0) leaves w'^2, the error of a zero dequant
#pragma unroll 4
  for (int p = 0; p < GS / 2; p += 2) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t wv = wt2[p + u][t];
      const float4 rc = rowc[p + u];
      const float2 wp = __fmul2_rn(make_float2(bf16lo(wv), bf16hi(wv)), make_float2(rc.x, rc.y));
      float2 r = __fadd2_rn(__ffma2_rn(wp, inv2, zm2), nzm2);
      const float2 dv = __ffma2_rn(wp, ninv2, r);
      dev = maxabs3f(dev, dv.x, dv.y);
      if (!SYM) {
        r.x = fminf(r.x, hic);
        r.y = fminf(r.y, hic);
      }
      const float2 d = __ffma2_rn(r, nstep2, wp);
      float2& acc = u ? acc1 : acc0;
      acc = __ffma2_rn(make_float2(rc.z, rc.w), __fmul2_rn(d, d), acc);
    }
  }
  if (dev > kTieGuard) {
    // exact form: clamp(rint(IEEE w'/step) + zero) - zero, same sums
    acc0 = acc1 = make_float2(0.f, 0.f);
    for (int p = 0; p < GS / 2; p += 2) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t wv = wt2[p + u][t];
        const float4 rc = rowc[p + u];
        const float wp[2] = {__fmul_rn(bf16lo(wv), rc.x), __fmul_rn(bf16hi(wv), rc.y)};
        float d[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float c = 0.f;
          if (q.step != 0.f) {
            const float tq = rintf(__fdiv_rn(wp[h], q.step));
            c = SYM ? fminf(fmaxf(tq, -7.f), 7.f) : fminf(fmaxf(tq + q.zero, 0.f), 15.f) - q.zero;
          }
          d[h] = fmaf(-c, q.step, wp[h]);
        }
        float2& acc = u ? acc1 : acc0;
        acc = __ffma2_rn(make_float2(rc.z, rc.w), make_float2(d[0] * d[0], d[1] * d[1]), acc);
      }
    }
  }
  return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

template <bool SYM>
__device__ __forceinline__ Range widen(Range r, float wp) {
  if (SYM) {
    r.hi = fmaxf(r.hi, fabsf(wp));
  } else {
    r.lo = fminf(r.lo, wp);
    r.hi = fmaxf(r.hi, wp);
  }
  return r;
}

// a fixed-order warp sum of v; lane 0 stores it
__device__ __forceinline__ void warp_sum_to(float v, float* dst, int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  if (lane == 0) *dst = v;
}

template <int GS, bool SYM>
__global__ void __launch_bounds__(kGreedyCols)
    greedy_step_kernel(const __nv_bfloat16* __restrict__ W, const float* __restrict__ a, int64_t D_out, int jj,
                       int pass, int k_min, int ncand, float* __restrict__ s_cur, int* __restrict__ cur_idx,
                       float* __restrict__ partial, unsigned int* __restrict__ tickets, int* __restrict__ trace,
                       double* __restrict__ errors, int64_t D_in, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t dyn[];
  uint32_t (*wt2)[kGreedyCols] = reinterpret_cast<uint32_t (*)[kGreedyCols]>(dyn);  // [GS / 2][128] row pairs
  __shared__ float4 rowc[GS / 2];
  // per warp: the column sum of each candidate's error change against the
  // common part, and (entry kMaxGreedyCand) of the common part itself, the
  // other rows' error under the range without channel jj
  __shared__ float red[kGreedyCols / 32][kMaxGreedyCand + 1];
  __shared__ bool last;

  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int g = blockIdx.y;
  const int slices = gridDim.x;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kGreedyCols;
  const int64_t row0 = static_cast<int64_t>(g) * GS;
  const bool active = n0 + t < D_out;

  // the group's rows of this column slice as row pairs, 16 bytes per load
  // (zeros past D_out, a multiple of 8: they add nothing)
  for (int v = t; v < (GS / 2) * (kGreedyCols / 8); v += kGreedyCols) {
    const int p = v / (kGreedyCols / 8), c8 = (v % (kGreedyCols / 8)) * 8;
    uint4 e = make_uint4(0u, 0u, 0u, 0u), o = e;
    if (n0 + c8 < D_out) {
      e = *reinterpret_cast<const uint4*>(W + (row0 + 2 * p) * D_out + n0 + c8);
      o = *reinterpret_cast<const uint4*>(W + (row0 + 2 * p + 1) * D_out + n0 + c8);
    }
    uint4* dst = reinterpret_cast<uint4*>(&wt2[p][c8]);
    dst[0] = make_uint4(__byte_perm(e.x, o.x, 0x5410), __byte_perm(e.x, o.x, 0x7632), __byte_perm(e.y, o.y, 0x5410),
                        __byte_perm(e.y, o.y, 0x7632));
    dst[1] = make_uint4(__byte_perm(e.z, o.z, 0x5410), __byte_perm(e.z, o.z, 0x7632), __byte_perm(e.w, o.w, 0x5410),
                        __byte_perm(e.w, o.w, 0x7632));
  }
  for (int p = t; p < GS / 2; p += kGreedyCols) {
    const int i = 2 * p;
    const float s0 = s_cur[row0 + i], s1 = s_cur[row0 + i + 1];
    const float r0 = 1.f / s0, r1 = 1.f / s1;  // exact: powers of two
    rowc[p] = make_float4(s0, s1, i == jj ? 0.f : a[row0 + i] * r0 * r0, i + 1 == jj ? 0.f : a[row0 + i + 1] * r1 * r1);
  }
  __syncthreads();
  // each thread reads only its own column: take channel jj's weight and leave
  // a zero in its place (a zero weight changes no range and adds no error)
  const uint32_t wjj = wt2[jj >> 1][t];
  const float wj = (jj & 1) ? bf16hi(wjj) : bf16lo(wjj);
  wt2[jj >> 1][t] = (jj & 1) ? (wjj & 0x0000FFFFu) : (wjj & 0xFFFF0000u);

  // range of the column without channel jj
  Range ex;
  ex.lo = 0.f;
  ex.hi = 0.f;
#pragma unroll 8
  for (int p = 0; p < GS / 2; ++p) {
    const uint32_t wv = wt2[p][t];
    const float4 rc = rowc[p];
    const float2 wp = __fmul2_rn(make_float2(bf16lo(wv), bf16hi(wv)), make_float2(rc.x, rc.y));
    if (SYM) {
      ex.hi = maxabs3f(ex.hi, wp.x, wp.y);
    } else {
      ex.lo = min3f(ex.lo, wp.x, wp.y);
      ex.hi = max3f(ex.hi, wp.x, wp.y);
    }
  }
  const Quant qb = quant_of<SYM>(ex, status);
  const float base = active ? column_error<GS, SYM>(wt2, rowc, t, qb) : 0.f;
  warp_sum_to(base, &red[warp][kMaxGreedyCand], lane);
  const float aj = a[row0 + jj];
#pragma unroll 1
  for (int c = 0; c < ncand; ++c) {
    const float sc = ldexpf(1.f, k_min + c);
    const float v = wj * sc;  // exact
    float e = 0.f;            // change of the column's error against the common part
    if (active) {
      const bool wider = SYM ? fabsf(v) > ex.hi : (v < ex.lo || v > ex.hi);
      const Quant q = wider ? quant_of<SYM>(widen<SYM>(ex, v), status) : qb;
      if (q.step != qb.step || q.zero != qb.zero) e = column_error<GS, SYM>(wt2, rowc, t, q) - base;
      float dev = 0.f;
      float own = term<SYM, false>(wj, sc, 1.f / sc, aj, q, dev);
      if (dev > kTieGuard) own = term<SYM, true>(wj, sc, 1.f / sc, aj, q, dev);
      e += own;
    }
    warp_sum_to(e, &red[warp][c], lane);
  }
  __syncthreads();
  if (t < ncand || t == kMaxGreedyCand) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kGreedyCols / 32; ++w) v += red[w][t];
    partial[(static_cast<int64_t>(g) * slices + blockIdx.x) * (kMaxGreedyCand + 1) + t] = v;
  }
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&tickets[g], 1u) == static_cast<unsigned>(slices) - 1u;
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (t < 32) {
    // lane c: the group's error change for candidate c, and the common part,
    // each summed over the slices in order; the decision compares changes
    const float* pg = partial + static_cast<int64_t>(g) * slices * (kMaxGreedyCand + 1);
    double e = 0.0, common = 0.0;
    for (int s0 = 0; s0 < slices; s0 += 16) {
      float v[16], b[16];  // 16 slices' loads in flight, added in slice order
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const bool in = s0 + i < slices;
        v[i] = in && t < ncand ? pg[(s0 + i) * (kMaxGreedyCand + 1) + t] : 0.f;
        b[i] = in && errors ? pg[(s0 + i) * (kMaxGreedyCand + 1) + kMaxGreedyCand] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        e += static_cast<double>(v[i]);
        common += static_cast<double>(b[i]);
      }
    }
    const int64_t j = row0 + jj;
    if (errors && t < ncand) errors[(static_cast<int64_t>(pass) * D_in + j) * ncand + t] = common + e;
    // strictly better than the current scale; the first in k order among equals
    const int cur = cur_idx[j];
    double best_e = __shfl_sync(0xFFFFFFFFu, e, cur);
    int best = cur;
    for (int c = 0; c < ncand; ++c) {
      const double ec = __shfl_sync(0xFFFFFFFFu, e, c);
      if (ec < best_e) {
        best_e = ec;
        best = c;
      }
    }
    if (t == 0) {
      cur_idx[j] = best;
      s_cur[j] = ldexpf(1.f, k_min + best);
      if (trace) trace[static_cast<int64_t>(pass) * D_in + j] = best;
      tickets[g] = 0u;  // ready for the next launch
    }
  }
}

__global__ void greedy_init_kernel(int64_t D_in, int idx_one, float* s_cur, int* cur_idx) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j < D_in) {
    s_cur[j] = 1.f;
    cur_idx[j] = idx_one;
  }
}

template <int GS, bool SYM>
cudaError_t run_greedy_t(const void* W, const float* a, int64_t D_in, int64_t D_out, int passes, int k_min,
                         int ncand, float* s_cur, int* cur_idx, float* partial, unsigned int* tickets, int* trace,
                         double* errors, uint32_t* status, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((D_out + kGreedyCols - 1) / kGreedyCols), static_cast<unsigned>(D_in / GS));
  const int smem = GS * kGreedyCols * 2;
  cudaError_t e0 = cudaFuncSetAttribute(greedy_step_kernel<GS, SYM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e0 != cudaSuccess) return e0;
  for (int p = 0; p < passes; ++p) {
    for (int jj = 0; jj < GS; ++jj) {
      greedy_step_kernel<GS, SYM><<<grid, kGreedyCols, smem, stream>>>(
          static_cast<const __nv_bfloat16*>(W), a, D_out, jj, p, k_min, ncand, s_cur, cur_idx, partial, tickets,
          trace, errors, D_in, status);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace

int64_t greedy_slices(int64_t D_out) { return (D_out + kGreedyCols - 1) / kGreedyCols; }

cudaError_t launch_greedy(const void* W, const float* a, int64_t D_in, int64_t D_out, int group_size, int symmetric,
                          int passes, int k_min, int ncand, float* s_cur, int* cur_idx, float* partial,
                          unsigned int* tickets, int* trace, double* errors, uint32_t* status, cudaStream_t stream) {
  const int idx_one = -k_min;
  greedy_init_kernel<<<static_cast<unsigned>((D_in + 255) / 256), 256, 0, stream>>>(D_in, idx_one, s_cur, cur_idx);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
#define AWQ_GREEDY(GS)                                                                                          \
  return symmetric ? run_greedy_t<GS, true>(W, a, D_in, D_out, passes, k_min, ncand, s_cur, cur_idx, partial,   \
                                            tickets, trace, errors, status, stream)                             \
                   : run_greedy_t<GS, false>(W, a, D_in, D_out, passes, k_min, ncand, s_cur, cur_idx, partial,  \
                                             tickets, trace, errors, status, stream)
  switch (group_size) {
    case 64:
      AWQ_GREEDY(64);
    case 128:
      AWQ_GREEDY(128);
    case 256:
      AWQ_GREEDY(256);
    default:
      return cudaErrorInvalidValue;
  }
#undef AWQ_GREEDY
}

}  // namespace awqdev
