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
// HBM-bound streaming kernel.  A persistent CTA walks tiles of one group
// (GS rows) x 8192/GS columns (16 KB of W).  TMA loads of the W tile and the
// group's slice of s run 3 tiles ahead in a ring; four warps take each tile
// from shared memory, and four such CTAs share an SM so that one CTA's
// serial step / zero phase overlaps the others' arithmetic.  A compute thread owns 8 columns
// and 4 row pairs, so both rows of a packed byte sit in one thread.  Pass 1
// finds the per-column range (shuffles over the row slots of a warp, then
// the 4 warps in a fixed order in shared memory) and the exact step / zero;
// pass 2 emits codes.
//
// Codes equal clamp(rint(fp32(w'/step)) + zero): the quotient is first
// formed as w' * (1/step); where that lands within 8e-6 of a half-integer
// (where the two could round differently), the thread redoes its rows with
// the IEEE division.  |w'/step| <= 45 in every case, where the product is
// within 6e-6 of the IEEE quotient, so elsewhere both round alike.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {
namespace {

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kTieGuard = 0.5f - 8.0e-6f;
constexpr int kPackStages = 3;
constexpr int kComputeWarps = 4;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kPackThreads = kComputeThreads;
constexpr int kRowsPerThread = 8;                   // four row pairs

// A tile is one group (GS rows) x COLS columns, 16 KB of W for every GS:
// 128 threads = CHUNKS 8-column chunks x PSLOTS row-pair slots.
template <int GS>
struct PackTile {
  static constexpr int PSLOTS = GS / kRowsPerThread;
  static constexpr int CHUNKS = kComputeThreads / PSLOTS;
  static constexpr int COLS = CHUNKS * 8;
  static constexpr int kWBytes = GS * COLS * 2;
  static constexpr int kSBytes = GS * 4;
  static constexpr int kStageBytes = kWBytes + kSBytes;  // a multiple of 128
  static constexpr int PAD = 12;                         // floats per chunk of column data (bank spread)
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
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

template <int GS, bool SYM>
__global__ void __launch_bounds__(kPackThreads, 4)
    pack_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS, int64_t D_in,
                int64_t D_out, uint8_t* __restrict__ qweight, __half* __restrict__ scales, __half* __restrict__ zeros,
                uint32_t* status) {
  using Tl = PackTile<GS>;
  constexpr int CH = Tl::CHUNKS, PS = Tl::PSLOTS, COLS = Tl::COLS, PAD = Tl::PAD;
  constexpr int SLOTS_PER_WARP = 32 / CH > 0 ? 32 / CH : 1;  // row-pair slots inside one warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ __align__(8) uint64_t full_bar[kPackStages];
  // per-tile column data in 8-column chunks padded to 12 floats, so that the
  // 8 chunks read by a quarter-warp fall on disjoint banks
  __shared__ __align__(16) float red_lo[kComputeWarps][CH * PAD];
  __shared__ __align__(16) float red_hi[kComputeWarps][CH * PAD];
  __shared__ __align__(16) float prm_inv[CH * PAD];
  __shared__ __align__(16) float prm_zoff[CH * PAD];
  __shared__ __align__(16) float prm_step[CH * PAD];
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nb = static_cast<int>((D_out + COLS - 1) / COLS);
  const int num_tiles = static_cast<int>(D_in / GS) * nb;
  volatile int* abort_flag = &abort_sh;
  // Thread 0 loads tile j (the CTA's j-th) into stage j % kPackStages: the
  // first kPackStages up front, then tile i + kPackStages - 1 at the top of
  // iteration i, right after the barrier that ends every read of the stage
  // tile i - 1 used.
  auto issue = [&](int j) {
    const int tile = blockIdx.x + j * gridDim.x;
    if (tile >= num_tiles) return;
    const int s = j % kPackStages;
    const int grp = tile / nb;
    const int cb = tile - grp * nb;
    uint8_t* st = smem + s * Tl::kStageBytes;
    mbar_arrive_expect_tx(&full_bar[s], Tl::kStageBytes);
    tma_load_2d(st, &tmW, &full_bar[s], cb * COLS, grp * GS);
    tma_load_2d(st + Tl::kWBytes, &tmS, &full_bar[s], grp * GS, 0);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPackStages; ++s) mbar_init(&full_bar[s], 1);
    abort_sh = 0;
    fence_mbar_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmS);
    for (int j = 0; j < kPackStages; ++j) issue(j);
  }
  __syncthreads();

  // -------------------------------------------------------------- compute warps
  // thread t: chunk c = t % CH (columns 8c .. 8c+7 of the tile), row-pair
  // slot p = t / CH: rows 2p + 2*PS*i and 2p + 2*PS*i + 1, i < 4
  const int t = threadIdx.x;
  const int c = t % CH;
  const int pslot = t / CH;
  int i = 0;
  for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++i) {
    const int s = i % kPackStages;
    const bool ok = mbar_wait(&full_bar[s], (i / kPackStages) & 1, status, abort_flag);
    if (named_bar_or(1, kComputeThreads, !ok)) {
      // loads still in flight into this CTA land before it exits
      // (tiles i .. i + kPackStages - 2 were issued, or 0 .. kPackStages - 1 when i == 0)
      if (threadIdx.x == 0) {
        const int last = i == 0 ? kPackStages : i + kPackStages - 1;
        for (int j = i; j < last && blockIdx.x + j * gridDim.x < num_tiles; ++j)
          mbar_wait(&full_bar[j % kPackStages], (j / kPackStages) & 1, nullptr, nullptr);
      }
      break;
    }
    if (threadIdx.x == 0 && i > 0) issue(i + kPackStages - 1);
    const int grp = tile / nb;
    const int cb = tile - grp * nb;
    const int64_t n = static_cast<int64_t>(cb) * COLS + c * 8;
    const bool active = n < D_out;
    const uint8_t* st = smem + s * Tl::kStageBytes;
    const float* ssl = reinterpret_cast<const float*>(st + Tl::kWBytes);

    // row r of this thread is 2p + 2*PS*(r/2) + r%2; both passes read the
    // rows from the stage, which stays in place until the codes are written
    const uint8_t* wbase = st + (2 * pslot) * (COLS * 2) + c * 16;
    const float* sbase = ssl + 2 * pslot;
#define PACK_WROW(r) (*reinterpret_cast<const uint4*>(wbase + (((r) & 1) + 2 * PS * ((r) >> 1)) * (COLS * 2)))
#define PACK_SROW(r) (sbase[((r) & 1) + 2 * PS * ((r) >> 1)])

    // pass 1: per-column range of w' = w * s (two rows per step: packed
    // products, three-input min / max); columns past D_out hold zeros
    float lo[8], hi[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) lo[k] = hi[k] = 0.f;
#pragma unroll
    for (int r = 0; r < kRowsPerThread; r += 2) {
      const uint4 a = PACK_WROW(r), b = PACK_WROW(r + 1);
      const float sa = PACK_SROW(r), sb = PACK_SROW(r + 1);
      const uint32_t we[4] = {a.x, a.y, a.z, a.w};
      const uint32_t wo[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 pe = __fmul2_rn(make_float2(bf16lo(we[k]), bf16hi(we[k])), make_float2(sa, sa));
        const float2 po = __fmul2_rn(make_float2(bf16lo(wo[k]), bf16hi(wo[k])), make_float2(sb, sb));
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
    // row slots of one warp that share a chunk: lanes l ^ CH, l ^ 2CH, ...
#pragma unroll
    for (int off = CH; off < 32; off <<= 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (!SYM) lo[k] = nmin(lo[k], __shfl_xor_sync(0xFFFFFFFFu, lo[k], off));
        hi[k] = nmax(hi[k], __shfl_xor_sync(0xFFFFFFFFu, hi[k], off));
      }
    }
    static_assert(SLOTS_PER_WARP * CH == 32 || CH == 32, "chunks tile a warp");
    if (lane < (CH < 32 ? CH : 32)) {
      float4* dh = reinterpret_cast<float4*>(&red_hi[warp][c * PAD]);
      dh[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
      dh[1] = make_float4(hi[4], hi[5], hi[6], hi[7]);
      if (!SYM) {
        float4* dl = reinterpret_cast<float4*>(&red_lo[warp][c * PAD]);
        dl[0] = make_float4(lo[0], lo[1], lo[2], lo[3]);
        dl[1] = make_float4(lo[4], lo[5], lo[6], lo[7]);
      }
    }
    named_bar_sync(1, kComputeThreads);
    if (t < COLS) {
      // exact step / zero of column t, the 4 warps combined in a fixed order
      const int col = t;
      const int pcol = (col >> 3) * PAD + (col & 7);
      float l = 0.f, h = 0.f;
#pragma unroll
      for (int k = 0; k < kComputeWarps; ++k) {
        if (!SYM) l = nmin(l, red_lo[k][pcol]);
        h = nmax(h, red_hi[k][pcol]);
      }
      float sc = 0.f;
      if (!isfinite(l) || !isfinite(h)) {
        set_error(status, AWQ_DEV_NONFINITE);  // codes of this column stay 0 (or 8)
      } else {
        const float raw = SYM ? __fdiv_rn(h, 7.0f) : __fdiv_rn(__fsub_rn(h, l), 15.0f);
        sc = __half2float(__float2half_rn(raw));
        if (isinf(sc)) {
          set_error(status, AWQ_DEV_RANGE);
          sc = 0.f;
        }
      }
      float z = 0.f;
      // an integer code in [0, 15]; the int round trip also turns -0 into +0
      if (!SYM && sc != 0.f) z = static_cast<float>(static_cast<int>(fminf(fmaxf(rintf(__fdiv_rn(-l, sc)), 0.f), 15.f)));
      prm_step[pcol] = sc;
      prm_inv[pcol] = sc != 0.f ? __frcp_rn(sc) : 0.f;
      prm_zoff[pcol] = SYM ? 8.f : z;
      const int64_t ncol = static_cast<int64_t>(cb) * COLS + col;
      if (ncol < D_out) {
        scales[grp * D_out + ncol] = __float2half_rn(sc);
        zeros[grp * D_out + ncol] = __float2half_rn(SYM ? 8.f : z);
      }
    }
    named_bar_sync(1, kComputeThreads);
    if (!active) continue;

    float inv[8], zmz[8];
    {
      const float4* pi = reinterpret_cast<const float4*>(prm_inv + c * PAD);
      const float4* pz = reinterpret_cast<const float4*>(prm_zoff + c * PAD);
      const float4 i0 = pi[0], i1 = pi[1], z0 = pz[0], z1 = pz[1];
      const float ia[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
      const float za[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        inv[k] = ia[k];
        zmz[k] = kMagic + za[k];
      }
    }
    // code range as 1.5*2^23 + code.  Asymmetric codes cannot fall below 0
    // on the fast path: rint is odd, so the group minimum gets
    // rint(min/step) + rint(-min/step) = 0 and every other element more.
    const float clo = SYM ? kMagic + 1.f : kMagic;
    const float chi = kMagic + 15.f;

    // pass 2 (fast): codes through the reciprocal.  c = fma(w', 1/step,
    // 1.5*2^23 + zero) rounds the exact product to an integer code; d =
    // rint - w'/step (one more fma) is within 1/2 of it, and tmax, the largest
    // |d|, flags a near tie anywhere in the thread's elements.  Each packed
    // byte is c_even + 16 c_odd in the low bits (1.5*2^23 has a zero low byte).
    uint32_t out[kRowsPerThread / 2][2];
    float tmax = 0.f;
#pragma unroll
    for (int p = 0; p < kRowsPerThread / 2; ++p) {
      const uint4 a = PACK_WROW(2 * p), b = PACK_WROW(2 * p + 1);
      const float se = PACK_SROW(2 * p), so = PACK_SROW(2 * p + 1);
      const uint32_t we[4] = {a.x, a.y, a.z, a.w};
      const uint32_t wo[4] = {b.x, b.y, b.z, b.w};
      uint32_t half16[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 inv2 = make_float2(inv[2 * k], inv[2 * k + 1]);
        const float2 ninv2 = make_float2(-inv[2 * k], -inv[2 * k + 1]);
        const float2 zm2 = make_float2(zmz[2 * k], zmz[2 * k + 1]);
        const float2 nzm2 = make_float2(-zmz[2 * k], -zmz[2 * k + 1]);
        const float2 pe = __fmul2_rn(make_float2(bf16lo(we[k]), bf16hi(we[k])), make_float2(se, se));
        const float2 po = __fmul2_rn(make_float2(bf16lo(wo[k]), bf16hi(wo[k])), make_float2(so, so));
        float2 ce = __ffma2_rn(pe, inv2, zm2);
        float2 co = __ffma2_rn(po, inv2, zm2);
        const float2 de = __ffma2_rn(pe, ninv2, __fadd2_rn(ce, nzm2));
        const float2 dd = __ffma2_rn(po, ninv2, __fadd2_rn(co, nzm2));
        tmax = maxabs3(tmax, de.x, de.y);
        tmax = maxabs3(tmax, dd.x, dd.y);
        if (SYM) {
          ce.x = fmaxf(ce.x, clo);
          ce.y = fmaxf(ce.y, clo);
          co.x = fmaxf(co.x, clo);
          co.y = fmaxf(co.y, clo);
        }
        ce.x = fminf(ce.x, chi);
        ce.y = fminf(ce.y, chi);
        co.x = fminf(co.x, chi);
        co.y = fminf(co.y, chi);
        const uint32_t x0 = __float_as_uint(co.x) * 16u + __float_as_uint(ce.x);  // byte 2k in the low 8 bits
        const uint32_t x1 = __float_as_uint(co.y) * 16u + __float_as_uint(ce.y);  // byte 2k+1
        half16[k] = __byte_perm(x0, x1, 0x0040);
      }
      out[p][0] = __byte_perm(half16[0], half16[1], 0x5410);
      out[p][1] = __byte_perm(half16[2], half16[3], 0x5410);
    }
    if (tmax > kTieGuard) {
      // slow path: IEEE quotient for every element of this thread
      float step[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) step[k] = prm_step[c * PAD + k];
#pragma unroll
      for (int p = 0; p < kRowsPerThread / 2; ++p) {
        const uint4 a = PACK_WROW(2 * p), b = PACK_WROW(2 * p + 1);
        const float se = PACK_SROW(2 * p), so = PACK_SROW(2 * p + 1);
        const uint32_t we[4] = {a.x, a.y, a.z, a.w};
        const uint32_t wo[4] = {b.x, b.y, b.z, b.w};
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
            const float qe = rintf(__fdiv_rn(__fmul_rn(xe, se), step[k])) + zo;
            const float qo = rintf(__fdiv_rn(__fmul_rn(xo, so), step[k])) + zo;
            ke = static_cast<uint32_t>(fminf(fmaxf(qe, ql), 15.f));
            ko = static_cast<uint32_t>(fminf(fmaxf(qo, ql), 15.f));
          }
          bytes[k] = ke | (ko << 4);
        }
        out[p][0] = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
        out[p][1] = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
      }
    }
#pragma unroll
    for (int p = 0; p < kRowsPerThread / 2; ++p) {
      const int64_t prow = (static_cast<int64_t>(grp) * GS + 2 * pslot + 2 * PS * p) / 2;
      *reinterpret_cast<uint2*>(qweight + prow * D_out + n) = make_uint2(out[p][0], out[p][1]);
    }
#undef PACK_WROW
#undef PACK_SROW
  }
}

cudaError_t encode_2d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, CUtensorMapDataType dt,
                      const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                      uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int GS, bool SYM>
cudaError_t launch_pack_t(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* W, const float* s, int64_t D_in,
                          int64_t D_out, uint8_t* qweight, void* scales, void* zeros, uint32_t* status, int num_sms,
                          cudaStream_t stream) {
  using Tl = PackTile<GS>;
  CUtensorMap tmW, tmS;
  cudaError_t e = encode_2d(encode, &tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, static_cast<uint64_t>(D_out),
                            static_cast<uint64_t>(D_in), static_cast<uint64_t>(D_out) * 2, Tl::COLS, GS);
  if (e != cudaSuccess) return e;
  e = encode_2d(encode, &tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, s, static_cast<uint64_t>(D_in), 1,
                static_cast<uint64_t>(D_in) * 4, GS, 1);
  if (e != cudaSuccess) return e;
  const int smem = kPackStages * Tl::kStageBytes + 128;  // + alignment slack
  e = cudaFuncSetAttribute(pack_kernel<GS, SYM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pack_kernel<GS, SYM>, kPackThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t tiles = (D_in / GS) * ((D_out + Tl::COLS - 1) / Tl::COLS);
  int64_t grid = static_cast<int64_t>(per_sm) * num_sms;
  if (grid > tiles) grid = tiles;
  pack_kernel<GS, SYM><<<static_cast<unsigned>(grid), kPackThreads, smem, stream>>>(
      tmW, tmS, D_in, D_out, qweight, static_cast<__half*>(scales), static_cast<__half*>(zeros), status);
  return cudaGetLastError();
}

template <int GS>
cudaError_t launch_pack_g(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* W, const float* s, int64_t D_in,
                          int64_t D_out, int symmetric, uint8_t* qweight, void* scales, void* zeros, uint32_t* status,
                          int num_sms, cudaStream_t stream) {
  if (symmetric)
    return launch_pack_t<GS, true>(encode, W, s, D_in, D_out, qweight, scales, zeros, status, num_sms, stream);
  return launch_pack_t<GS, false>(encode, W, s, D_in, D_out, qweight, scales, zeros, status, num_sms, stream);
}


// ---------------------------------------------------------------------------
// Pack after a search.  The search's group-parameter pass already holds, for
// every candidate, the exact step (fp16-rounded range / 15 or max|w'| / 7),
// 1/step and zero of every (group, column) -- the same formulas and the same
// exact ranges as pass 1 above.  For its best candidate the pack is then a
// single streaming pass: thread t of the grid owns 8 columns (chunk c) x 8
// rows of one group, loads all 8 rows at once, and emits codes exactly as
// pass 2 above (with the same exact-division redo near ties); the threads
// of chunk-0-row-block write the group's fp16 scales and zeros.
constexpr int kSearchedRows = 8;
constexpr int kSearchedThreads = 256;

// The exact path of one thread's 8 rows x 8 columns (rare: only where some
// quotient lies within the tie guard of a half step): codes from the IEEE
// fp32 quotient w'/step, as the oracle defines them.  Kept out of line so
// that its registers do not burden the streaming path.
template <bool SYM>
__device__ __noinline__ void pack_searched_exact(const __nv_bfloat16* __restrict__ W, const float* __restrict__ s,
                                                 const float* __restrict__ qc, int64_t row0, int64_t n,
                                                 int64_t D_out, uint8_t* __restrict__ qweight) {
  for (int p = 0; p < kSearchedRows / 2; ++p) {
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

template <int GS, bool SYM>
__global__ void __launch_bounds__(kSearchedThreads, 3)
    pack_searched_kernel(const __nv_bfloat16* __restrict__ W, const float* __restrict__ s,
                         const float* __restrict__ qp, const int32_t* __restrict__ best_idx, int G, int64_t D_in,
                         int64_t D_out, uint8_t* __restrict__ qweight, __half* __restrict__ scales,
                         __half* __restrict__ zeros) {
  constexpr int RB = GS / kSearchedRows;  // row blocks per group
  const int64_t chunks = D_out / kQChunkCols;
  const int64_t T = D_in / GS;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * kSearchedThreads + threadIdx.x;
  if (idx >= T * RB * chunks) return;
  const int64_t c = idx % chunks;  // chunk fastest: a warp reads 512 contiguous bytes per row
  const int64_t rest = idx / chunks;
  const int rb = static_cast<int>(rest % RB);
  const int64_t g = rest / RB;
  const int64_t n = c * kQChunkCols;
  const int64_t row0 = g * GS + rb * kSearchedRows;

  uint4 w[kSearchedRows];
#pragma unroll
  for (int i = 0; i < kSearchedRows; ++i) w[i] = *reinterpret_cast<const uint4*>(W + (row0 + i) * D_out + n);
  float sj[kSearchedRows];
#pragma unroll
  for (int i = 0; i < kSearchedRows; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(s + row0 + i);  // rows of a group: 16-byte aligned
    sj[i] = v.x;
    sj[i + 1] = v.y;
    sj[i + 2] = v.z;
    sj[i + 3] = v.w;
  }
  // {1/step x8, 1.5*2^23 + zero x8, step x8} of (best candidate, group, chunk)
  int k = *best_idx;
  k = k < 0 ? 0 : (k >= G ? G - 1 : k);  // awq_search always writes an index in [0, G)
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
  if (rb == 0) {
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
  const float clo = SYM ? kMagic + 1.f : kMagic;
  const float chi = kMagic + 15.f;
  uint32_t out[kSearchedRows / 2][2];
  float tmax = 0.f;
#pragma unroll
  for (int p = 0; p < kSearchedRows / 2; ++p) {
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
      const float2 po = __fmul2_rn(make_float2(bf16lo(wo[j]), bf16hi(wo[j])), make_float2(sj[2 * p + 1], sj[2 * p + 1]));
      float2 ce = __ffma2_rn(pe, inv2, zm2);
      float2 co = __ffma2_rn(po, inv2, zm2);
      const float2 de = __ffma2_rn(pe, ninv2, __fadd2_rn(ce, nzm2));
      const float2 dd = __ffma2_rn(po, ninv2, __fadd2_rn(co, nzm2));
      tmax = maxabs3(tmax, de.x, de.y);
      tmax = maxabs3(tmax, dd.x, dd.y);
      if (SYM) {
        ce.x = fmaxf(ce.x, clo);
        ce.y = fmaxf(ce.y, clo);
        co.x = fmaxf(co.x, clo);
        co.y = fmaxf(co.y, clo);
      }
      ce.x = fminf(ce.x, chi);
      ce.y = fminf(ce.y, chi);
      co.x = fminf(co.x, chi);
      co.y = fminf(co.y, chi);
      const uint32_t x0 = __float_as_uint(co.x) * 16u + __float_as_uint(ce.x);
      const uint32_t x1 = __float_as_uint(co.y) * 16u + __float_as_uint(ce.y);
      half16[j] = __byte_perm(x0, x1, 0x0040);
    }
    out[p][0] = __byte_perm(half16[0], half16[1], 0x5410);
    out[p][1] = __byte_perm(half16[2], half16[3], 0x5410);
  }
  if (tmax > kTieGuard) {
    pack_searched_exact<SYM>(W, s, qc, row0, n, D_out, qweight);
    return;
  }
#pragma unroll
  for (int p = 0; p < kSearchedRows / 2; ++p)
    *reinterpret_cast<uint2*>(qweight + (row0 / 2 + p) * D_out + n) = make_uint2(out[p][0], out[p][1]);
}

template <int GS, bool SYM>
cudaError_t launch_pack_searched_t(const void* W, const float* s, const float* qp, const int32_t* best_idx, int G,
                                   int64_t D_in, int64_t D_out, uint8_t* qweight, void* scales, void* zeros,
                                   cudaStream_t stream) {
  const int64_t threads = (D_in / GS) * (GS / kSearchedRows) * (D_out / kQChunkCols);
  const int64_t blocks = (threads + kSearchedThreads - 1) / kSearchedThreads;
  pack_searched_kernel<GS, SYM><<<static_cast<unsigned>(blocks), kSearchedThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(W), s, qp, best_idx, G, D_in, D_out, qweight, static_cast<__half*>(scales),
      static_cast<__half*>(zeros));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* W, const float* s, int64_t D_in,
                        int64_t D_out, int group_size, int symmetric, uint8_t* qweight, void* scales, void* zeros,
                        uint32_t* status, int num_sms, cudaStream_t stream) {
  switch (group_size) {
    case 64:
      return launch_pack_g<64>(encode, W, s, D_in, D_out, symmetric, qweight, scales, zeros, status, num_sms, stream);
    case 128:
      return launch_pack_g<128>(encode, W, s, D_in, D_out, symmetric, qweight, scales, zeros, status, num_sms, stream);
    case 256:
      return launch_pack_g<256>(encode, W, s, D_in, D_out, symmetric, qweight, scales, zeros, status, num_sms, stream);
    default:
      return cudaErrorInvalidValue;
  }
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
