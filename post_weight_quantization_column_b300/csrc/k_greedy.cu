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
// which case it re-sums the column under the new step / zero.  Codes are
// rint of the IEEE quotient w'/step as the oracle defines them, formed as
// w' * (1/step) and redone with the division within 8e-6 of a half step (s
// is a power of two, so w s and step / s are exact).  Column errors are summed in a fixed order
// (a warp tree, then the warps in order), the slices of a group in slice
// order in fp64 by the last CTA of the group to finish (ticket counter),
// which also takes the decision and updates the scale.
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
};

// Within this distance of a half step the reciprocal product and the IEEE
// quotient can round differently: |w'/step| <= 15 (1 + 2^-11) here, where the
// product is within 2e-6 of the quotient.
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
  q.zero = (!SYM && sc != 0.f) ? fminf(fmaxf(rintf(__fdiv_rn(-r.lo, sc)), 0.f), 15.f) : 0.f;
  q.inv = sc != 0.f ? __frcp_rn(sc) : 0.f;
  return q;
}

// a * (w'hat / s - w)^2 for one weight w with scale s and rs = 1/s (powers of
// two).  The fast form takes rint(w' * (1/step)) and raises `dev` to the
// distance of that product from its rounding; where dev ends above the tie
// guard the caller redoes the column with the exact form (rint of the IEEE
// quotient).
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

// sum over the group's rows of one column (row jj zeroed with weight 0)
template <int GS, bool SYM>
__device__ __forceinline__ float column_error(const __nv_bfloat16 (*wt)[128], const float* ss, const float* sr,
                                              const float* sa, int t, Quant q) {
  // four interleaved partial sums (rows i mod 4), added in a fixed order
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, dev[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int i = 0; i < GS; i += 4) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      acc[u] += term<SYM, false>(__bfloat162float(wt[i + u][t]), ss[i + u], sr[i + u], sa[i + u], q, dev[u]);
  }
  if (fmaxf(fmaxf(dev[0], dev[1]), fmaxf(dev[2], dev[3])) > kTieGuard) {
    float d = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = 0.f;
    for (int i = 0; i < GS; i += 4)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        acc[u] += term<SYM, true>(__bfloat162float(wt[i + u][t]), ss[i + u], sr[i + u], sa[i + u], q, d);
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
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

template <int GS, bool SYM>
__global__ void __launch_bounds__(kGreedyCols)
    greedy_step_kernel(const __nv_bfloat16* __restrict__ W, const float* __restrict__ a, int64_t D_out, int jj,
                       int pass, int k_min, int ncand, float* __restrict__ s_cur, int* __restrict__ cur_idx,
                       float* __restrict__ partial, unsigned int* __restrict__ tickets, int* __restrict__ trace,
                       double* __restrict__ errors, int64_t D_in, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __nv_bfloat16 (*wt)[kGreedyCols] = reinterpret_cast<__nv_bfloat16 (*)[kGreedyCols]>(dyn);  // [GS][128]
  __shared__ float sa[GS], ss[GS], sr[GS];
  // per column: the error change of each candidate against the common part
  // (row kMaxGreedyCand: the common part itself, the other rows' error under
  // the range without channel jj)
  __shared__ float errs[kMaxGreedyCand + 1][kGreedyCols];
  __shared__ float red[kGreedyCols / 32][kMaxGreedyCand + 1];
  __shared__ bool last;

  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int g = blockIdx.y;
  const int slices = gridDim.x;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kGreedyCols;
  const int64_t row0 = static_cast<int64_t>(g) * GS;
  const int64_t n = n0 + t;
  const bool active = n < D_out;

  // the group's rows of this column slice, 16 bytes per load (zeros past
  // D_out, a multiple of 8: they add nothing)
  for (int v = t; v < GS * (kGreedyCols / 8); v += kGreedyCols) {
    const int i = v / (kGreedyCols / 8), c8 = (v % (kGreedyCols / 8)) * 8;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (n0 + c8 < D_out) x = *reinterpret_cast<const uint4*>(W + (row0 + i) * D_out + n0 + c8);
    *reinterpret_cast<uint4*>(&wt[i][c8]) = x;
  }
  for (int i = t; i < GS; i += kGreedyCols) {
    sa[i] = i == jj ? 0.f : a[row0 + i];  // channel jj's own term is added per candidate
    ss[i] = s_cur[row0 + i];
    sr[i] = 1.f / ss[i];  // exact: a power of two
  }
  __syncthreads();
  // each thread reads only its own column: take channel jj's weight and leave
  // a zero in its place (a zero weight changes no range and adds no error)
  const float wj = __bfloat162float(wt[jj][t]);
  wt[jj][t] = __float2bfloat16(0.f);

  for (int c = 0; c <= kMaxGreedyCand; ++c) errs[c][t] = 0.f;
  if (active) {
    // range of the column without channel jj
    Range ex;
    ex.lo = 0.f;
    ex.hi = 0.f;
#pragma unroll 8
    for (int i = 0; i < GS; ++i) ex = widen<SYM>(ex, __bfloat162float(wt[i][t]) * ss[i]);
    const Quant qb = quant_of<SYM>(ex, status);
    const float base = column_error<GS, SYM>(wt, ss, sr, sa, t, qb);
    const float aj = a[row0 + jj];
#pragma unroll 1
    for (int c = 0; c < ncand; ++c) {
      const float sc = ldexpf(1.f, k_min + c);
      const Quant q = quant_of<SYM>(widen<SYM>(ex, wj * sc), status);
      float e = 0.f;  // change of the other rows' error
      if (q.step != qb.step || q.zero != qb.zero) e = column_error<GS, SYM>(wt, ss, sr, sa, t, q) - base;
      float dev = 0.f;
      float own = term<SYM, false>(wj, sc, 1.f / sc, aj, q, dev);
      if (dev > kTieGuard) own = term<SYM, true>(wj, sc, 1.f / sc, aj, q, dev);
      errs[c][t] = e + own;
    }
    errs[kMaxGreedyCand][t] = base;
  }
  // column sums per candidate: a warp tree, then the warps in order
  // (each thread reads back only its own column, so no barrier is needed yet)
  for (int c = 0; c <= kMaxGreedyCand; ++c) {
    if (c >= ncand && c < kMaxGreedyCand) continue;
    float v = errs[c][t];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == 0) red[warp][c] = v;
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
