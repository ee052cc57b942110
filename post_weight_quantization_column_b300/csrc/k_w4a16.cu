// W4A16 product on the packed layer (sm_103a), the online half of the pages'
// inference equivalence: Y = (X diag(1/s*)) Dequant(W_quantized), with the
// 1/s* scaling folded into the dequantisation ("AWQ (Activation-aware Weight
// Quantization)", 推理时的等效实现 and the pipeline figure's
// "Dequant + MatMul (融合 s* 缩放)"; Dequant = (code - zero) * scale,
// 量化数学基础 step 3).
//
// Same CTA-pair structure as the candidate search: a work unit is 512 rows of
// X x 256 columns of Y; each CTA of a cluster pair holds two stacked 128-row
// subtiles of X and produces the bf16 operand for 128 of the 256 columns; the
// even CTA issues M256 x N256 x K16 MMAs (fp32 accumulators in all 512 TMEM
// columns of both CTAs).  Per K step of 64 input rows the B operand is built
// in registers from the packed codes:
//   w_hat[j, n] = bf16( ((code - zero_n) * scale_n) * RN(1/s_j) )
// (code - zero) * scale is exact in fp32 (a 5-bit integer times an fp16
// value), so the only roundings are the product with 1/s_j and the bf16 cast.
//
// Roles (640 threads per CTA):
//   warp 0      TMA: X subtiles (K-major, 128-byte swizzle)
//   warp 1      TMEM allocation; in the even CTA the single-thread MMA issuer
//   warp 2      TMA: the step's 32 x 128 code bytes, the group's fp16 scales
//               and zeros of the CTA's 128 columns, and s of the 64 rows
//   warps 4-11  epilogue: TMEM -> registers -> bf16 -> Y
//   warps 12-19 producers: two groups of 4 warps on alternate K steps
//               (8 columns x 8 rows per thread per step)
// Every mbarrier wait is bounded; a timeout records AWQ_ERR_TIMEOUT and every
// role leaves its loop.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {
namespace {

constexpr int kBK = 64;                          // input rows per K step
constexpr int kSubRows = 128;
constexpr int kStack = 2;
constexpr int kPairN = 256;
constexpr int kHalfN = kPairN / 2;
constexpr int kAStages = 4;
constexpr int kBStages = 4;
constexpr int kASubBytes = kSubRows * kBK * 2;   // 16 KB
constexpr int kABytes = kStack * kASubBytes;     // 32 KB
constexpr int kBBytes = kBK * kHalfN * 2;        // 16 KB: 64 K x 128 N bf16, N-major, 128B swizzle
constexpr int kCodeBytes = (kBK / 2) * kHalfN;   // 4 KB: 32 byte rows x 128 columns
constexpr int kSBytes = kBK * 4;                 // s of the 64 rows
constexpr int kHBytes = kHalfN * 2;              // fp16 scales (or zeros) of 128 columns
constexpr int kSideTx = kCodeBytes + 2 * kHBytes;  // + kSBytes when s is given
constexpr int kSideStride = (kCodeBytes + kSBytes + 2 * kHBytes + 127) / 128 * 128;
constexpr int kOffB = kAStages * kABytes;
constexpr int kOffSide = kOffB + kBStages * kBBytes;
constexpr int kSmemBytes = kOffSide + kBStages * kSideStride;
constexpr int kTmemCols = 512;
constexpr int kThreads = 640;
constexpr int kEpiWarp0 = 4, kEpiWarps = 8;
constexpr int kProdWarp0 = 12, kProdWarps = 8;
constexpr int kGroupWarps = 4;
static_assert(kProdWarps == 2 * kGroupWarps, "two producer groups");
constexpr int kBFullCount = 2 * kGroupWarps;
constexpr int kAccEmptyCount = 2 * kEpiWarps;
static_assert(kSmemBytes + 1024 + 512 <= 227 * 1024, "shared memory (dynamic + alignment slack + static)");

struct GemmArgs {
  int M, D_in, D_out, group_size, has_s;
  int m_blocks, n_blocks, num_tiles;
  __nv_bfloat16* Y;
  uint32_t* status;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 2^23 + v for the four byte lanes of m (each byte < 16): byte k of m becomes
// the low byte of an fp32 whose high byte is 0x4B.
__device__ __forceinline__ void nibbles_to_f32(uint32_t m, float (&t)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) t[k] = __uint_as_float(__byte_perm(m, 0x4B000000u, 0x7650u | k));
}

struct Tile {
  int m_blk, n_blk;
};
__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs& p) {
  Tile r;
  r.n_blk = t % p.n_blocks;
  r.m_blk = t / p.n_blocks;
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    w4a16_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                 const __grid_constant__ CUtensorMap tmSc, const __grid_constant__ CUtensorMap tmZ,
                 const __grid_constant__ CUtensorMap tmS, GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t afull_bar[kAStages];   // even CTA: X of both CTAs landed
  __shared__ __align__(8) uint64_t aempty_bar[kAStages];  // both CTAs: MMAs done with the X slot
  __shared__ __align__(8) uint64_t cfull_bar[kBStages];   // local: codes and side inputs landed
  __shared__ __align__(8) uint64_t bfull_bar[kBStages];   // even CTA: B written by both CTAs
  __shared__ __align__(8) uint64_t bempty_bar[kBStages];  // both CTAs: MMAs done with the B slot
  __shared__ __align__(8) uint64_t acc_full_bar;
  __shared__ __align__(8) uint64_t acc_empty_bar;
  __shared__ __align__(8) uint64_t mma_drain_bar;          // even CTA: MMAs still running after an abort
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(nclusters_x());
  const int KB = p.D_in / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&afull_bar[s], 1);
      mbar_init(&aempty_bar[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&cfull_bar[s], 1);
      mbar_init(&bfull_bar[s], kBFullCount);
      mbar_init(&bempty_bar[s], 1);
    }
    mbar_init(&acc_full_bar, 1);
    mbar_init(&acc_empty_bar, kAccEmptyCount);
    mbar_init(&mma_drain_bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32 * 2) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmC);
    prefetch_tmap(&tmSc);
    prefetch_tmap(&tmZ);
    if (p.has_s) prefetch_tmap(&tmS);
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort_flag = &abort_sh;

  const uint32_t afull0 = mapa_shared(smem_u32(&afull_bar[0]), 0);
  const uint32_t bfull0 = mapa_shared(smem_u32(&bfull_bar[0]), 0);
  const uint32_t acc_empty0 = mapa_shared(smem_u32(&acc_empty_bar), 0);

  if (warp == 0) {
    // ---------------------------------------------------------- X loader
    if (lane == 0) {
      int it = 0;
      for (int t = pair; t < p.num_tiles && !*abort_flag; t += npairs) {
        const Tile tl = decode_tile(t, p);
        const int row0 = tl.m_blk * (2 * kStack * kSubRows) + static_cast<int>(rank) * kSubRows;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % kAStages;
          const uint32_t ph = (it / kAStages) & 1;
          if (it >= kAStages && !mbar_wait_cluster(&aempty_bar[s], ph ^ 1, p.status, abort_flag)) break;
          if (leader) mbar_arrive_expect_tx(&afull_bar[s], 2 * kABytes);
          const uint32_t bar = afull0 + static_cast<uint32_t>(s) * 8u;
#pragma unroll
          for (int sub = 0; sub < kStack; ++sub)
            tma_load_2d_pair(smem + s * kABytes + sub * kASubBytes, &tmX, bar, kb * kBK,
                             row0 + sub * 2 * kSubRows);
        }
        if (*abort_flag) break;
      }
      const int first = it - kAStages < 0 ? 0 : it - kAStages;
      for (int j = first; j < it; ++j)
        mbar_wait_cluster(&aempty_bar[j % kAStages], (j / kAStages) & 1, p.status, abort_flag);
      if (*abort_flag) {
        // after an abort those waits return at once: the X copies still in
        // flight land first.  Their completion is counted on the even CTA's
        // barriers, so the even CTA waits there (bounded: a phase the peer
        // never filled cannot complete) and the odd CTA gives them the same time.
        if (leader)
          for (int j = first; j < it; ++j)
            mbar_wait_cluster(&afull_bar[j % kAStages], (j / kAStages) & 1, nullptr, nullptr, kCopyDrainNs);
        else
          settle_ns(kCopyDrainNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (even CTA)
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(256, kPairN, 0, 1);
      int it = 0, tc = 0;
      for (int t = pair; t < p.num_tiles; t += npairs, ++tc) {
        if (tc > 0 && !mbar_wait_cluster(&acc_empty_bar, (tc - 1) & 1, p.status, abort_flag)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int sa = it % kAStages;
          const int sb = it % kBStages;
          if (!mbar_wait_cluster(&afull_bar[sa], (it / kAStages) & 1, p.status, abort_flag) ||
              !mbar_wait_cluster(&bfull_bar[sb], (it / kBStages) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + sa * kABytes);
          const uint32_t b_addr = smem_u32(smem + kOffB + sb * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(b_addr + kk * 2048, kBK * 128, 1024);
#pragma unroll
            for (int sub = 0; sub < kStack; ++sub) {
              const uint64_t ad = sdesc_sw128(a_addr + sub * kASubBytes + kk * 32, 16, 1024);
              umma_bf16_pair(tmem + static_cast<uint32_t>(sub * kPairN), ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit_pair_mc(&aempty_bar[sa], 0x3);
          umma_commit_pair_mc(&bempty_bar[sb], 0x3);
        }
        if (!ok) break;
        umma_commit_pair_mc(&acc_full_bar, 0x3);
      }
      if (tc > 0 && !*abort_flag) mbar_wait_cluster(&acc_empty_bar, (tc - 1) & 1, p.status, abort_flag);
      if (*abort_flag) {
        // no MMA of the pair may still run when TMEM is freed: one more
        // commit arrives once every MMA issued so far is done
        umma_commit_pair_mc(&mma_drain_bar, 0x1);
        mbar_wait(&mma_drain_bar, 0, nullptr, nullptr, kCopyDrainNs);
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- code / side-input loader
    if (lane == 0) {
      const uint32_t tx = kSideTx + (p.has_s ? kSBytes : 0);
      int it = 0;
      for (int t = pair; t < p.num_tiles && !*abort_flag; t += npairs) {
        const Tile tl = decode_tile(t, p);
        const int n_base = tl.n_blk * kPairN + static_cast<int>(rank) * kHalfN;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % kBStages;
          const uint32_t ph = (it / kBStages) & 1;
          if (it >= kBStages && !mbar_wait_cluster(&bempty_bar[s], ph ^ 1, p.status, abort_flag)) break;
          uint8_t* side = smem + kOffSide + s * kSideStride;
          const int grp = (kb * kBK) / p.group_size;
          mbar_arrive_expect_tx(&cfull_bar[s], tx);
          tma_load_2d(side, &tmC, &cfull_bar[s], n_base, kb * (kBK / 2));
          tma_load_2d(side + kCodeBytes, &tmSc, &cfull_bar[s], n_base, grp);
          tma_load_2d(side + kCodeBytes + kHBytes, &tmZ, &cfull_bar[s], n_base, grp);
          if (p.has_s) tma_load_2d(side + kCodeBytes + 2 * kHBytes, &tmS, &cfull_bar[s], kb * kBK, 0);
        }
        if (*abort_flag) break;
      }
      const int first = it - kBStages < 0 ? 0 : it - kBStages;
      for (int j = first; j < it; ++j)
        mbar_wait_cluster(&bempty_bar[j % kBStages], (j / kBStages) & 1, p.status, abort_flag);
      if (*abort_flag)  // after an abort: this CTA's own copies in flight land first
        for (int j = first; j < it; ++j)
          mbar_wait(&cfull_bar[j % kBStages], (j / kBStages) & 1, nullptr, nullptr, kCopyDrainNs);
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ---------------------------------------------------------- epilogue
    const int e = warp - kEpiWarp0;
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const int ch = e >> 2;    // column half
    int tc = 0;
    for (int t = pair; t < p.num_tiles; t += npairs, ++tc) {
      const Tile tl = decode_tile(t, p);
      const bool ok = mbar_wait(&acc_full_bar, tc & 1, p.status, abort_flag);
      tc_fence_after();
      if (!ok) break;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int i = 0; i < kStack * 4; ++i) {
        const int sub = i >> 2, cc = i & 3;
        const int col = ch * 128 + cc * 32;
        float a[32];
        tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(sub * kPairN + col), a);
        if (i == kStack * 4 - 1) {
          // every TMEM read of this warp is complete: release the accumulator
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acc_empty0);
        }
        const int64_t row = static_cast<int64_t>(tl.m_blk) * (2 * kStack * kSubRows) + sub * (2 * kSubRows) +
                            static_cast<int64_t>(rank) * kSubRows + q * 32 + lane;
        const int n0 = tl.n_blk * kPairN + col;
        if (row < p.M) {
          __nv_bfloat16* yrow = p.Y + row * p.D_out + n0;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (n0 + 8 * v < p.D_out) {
              const uint4 o = make_uint4(pack_bf16x2(a[8 * v], a[8 * v + 1]), pack_bf16x2(a[8 * v + 2], a[8 * v + 3]),
                                         pack_bf16x2(a[8 * v + 4], a[8 * v + 5]),
                                         pack_bf16x2(a[8 * v + 6], a[8 * v + 7]));
              *reinterpret_cast<uint4*>(yrow + 8 * v) = o;
            }
          }
        }
      }
      if (*abort_flag) break;
    }
  } else if (warp >= kProdWarp0) {
    // ---------------------------------------------------------- producers
    // Thread: 8 columns (chunk c of the CTA's 16) x 8 rows (byte rows
    // 4*rg .. 4*rg+3) of the 64 x 128 operand tile of its step.
    const int grp_id = (warp - kProdWarp0) / kGroupWarps;
    const int gt = threadIdx.x - (kProdWarp0 + grp_id * kGroupWarps) * 32;
    const int c = gt & 15;
    const int rg = gt >> 4;
    const int h = c >> 3;   // 64-column half of the CTA's 128 columns
    const int c8 = c & 7;   // 16-byte chunk inside a 128-byte row of the operand
    constexpr float kTwo23 = 8388608.0f;
    int it = 0;
    for (int t = pair; t < p.num_tiles && !*abort_flag; t += npairs) {
      int cached_group = -1;
      float2 zc2[4], sc2[4];  // per column pair: -(2^23 + zero), scale
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        if ((it & 1) != grp_id) continue;
        const int s = it % kBStages;
        if (!mbar_wait(&cfull_bar[s], (it / kBStages) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        // the B slot was released by the MMAs of step it - kBStages (the
        // loader waited for that release before it filled this stage)
        const uint8_t* side = smem + kOffSide + s * kSideStride;
        const int grp = (kb * kBK) / p.group_size;
        if (grp != cached_group) {
          cached_group = grp;
          const uint4 hs = *reinterpret_cast<const uint4*>(side + kCodeBytes + c * 16);
          const uint4 hz = *reinterpret_cast<const uint4*>(side + kCodeBytes + kHBytes + c * 16);
          const uint32_t us[4] = {hs.x, hs.y, hs.z, hs.w};
          const uint32_t uz[4] = {hz.x, hz.y, hz.z, hz.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            sc2[j] = __half22float2(*reinterpret_cast<const __half2*>(&us[j]));
            const float2 z = __half22float2(*reinterpret_cast<const __half2*>(&uz[j]));
            zc2[j] = make_float2(-(kTwo23 + z.x), -(kTwo23 + z.y));
          }
        }
        float r[8];
        if (p.has_s) {
          const float4* sp = reinterpret_cast<const float4*>(side + kCodeBytes + 2 * kHBytes) + rg * 2;
          const float4 s0 = sp[0], s1 = sp[1];
          r[0] = __frcp_rn(s0.x);
          r[1] = __frcp_rn(s0.y);
          r[2] = __frcp_rn(s0.z);
          r[3] = __frcp_rn(s0.w);
          r[4] = __frcp_rn(s1.x);
          r[5] = __frcp_rn(s1.y);
          r[6] = __frcp_rn(s1.z);
          r[7] = __frcp_rn(s1.w);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) r[i] = 1.f;
        }
        uint8_t* bslot = smem + kOffB + s * kBBytes + h * (kBK * 128) + (rg * 8) * 128;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
          // byte row 4*rg + pr holds input rows 8*rg + 2*pr (low nibbles) and 8*rg + 2*pr + 1
          const uint2 cb = *reinterpret_cast<const uint2*>(side + (rg * 4 + pr) * kHalfN + h * 64 + c8 * 8);
#pragma unroll
          for (int odd = 0; odd < 2; ++odd) {
            const int i = 2 * pr + odd;  // row inside the thread's 8
            float t[8];
            {
              float t0[4], t1[4];
              nibbles_to_f32(odd ? (cb.x >> 4) & 0x0F0F0F0Fu : cb.x & 0x0F0F0F0Fu, t0);
              nibbles_to_f32(odd ? (cb.y >> 4) & 0x0F0F0F0Fu : cb.y & 0x0F0F0F0Fu, t1);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                t[k] = t0[k];
                t[4 + k] = t1[k];
              }
            }
            const float2 r2 = make_float2(r[i], r[i]);
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 e2 = __fadd2_rn(make_float2(t[2 * j], t[2 * j + 1]), zc2[j]);  // code - zero, exact
              const float2 f2 = __fmul2_rn(e2, sc2[j]);                                   // * scale, exact
              const float2 w2 = __fmul2_rn(f2, r2);                                       // * 1/s_j
              o[j] = pack_bf16x2(w2.x, w2.y);
            }
            // row 8*rg + i of the slot: its 16-byte chunk c8 sits at c8 ^ (row & 7) = c8 ^ i
            *reinterpret_cast<uint4*>(bslot + i * 128 + ((c8 ^ i) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        fence_proxy_async_smem();  // stores visible to the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(bfull0 + static_cast<uint32_t>(s) * 8u);
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no arrival or MMA of one CTA may target an exited peer
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

cudaError_t encode_tiled(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, CUtensorMapDataType dt,
                         const void* base, cuuint64_t inner, cuuint64_t outer, cuuint64_t row_bytes,
                         cuuint32_t box_inner, cuuint32_t box_outer, CUtensorMapSwizzle sw) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaLaunchConfig_t pair_config(int pairs, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t w4a16_max_pairs(int* pairs) {
  const size_t smem = static_cast<size_t>(kSmemBytes) + 1024;
  cudaError_t e = cudaFuncSetAttribute(w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(1, smem, nullptr, attr);
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, w4a16_kernel, &cfg);
  if (e != cudaSuccess) return e;
  *pairs = n;
  return cudaSuccess;
}

cudaError_t launch_w4a16(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, int64_t M, int64_t D_in,
                         int64_t D_out, const uint8_t* qweight, const void* scales, const void* zeros, const float* s,
                         int group_size, void* Y, uint32_t* status, int max_pairs, cudaStream_t stream) {
  CUtensorMap tmX, tmC, tmSc, tmZ, tmS;
  const int T = static_cast<int>(D_in / group_size);
  cudaError_t e = encode_tiled(encode, &tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, D_in, M, D_in * 2, kBK, kSubRows,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = encode_tiled(encode, &tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, qweight, D_out, D_in / 2, D_out, kHalfN, kBK / 2,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = encode_tiled(encode, &tmSc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, scales, D_out, T, D_out * 2, kHalfN, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  e = encode_tiled(encode, &tmZ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, zeros, D_out, T, D_out * 2, kHalfN, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  if (s) {
    e = encode_tiled(encode, &tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, s, D_in, 1, D_in * 4, kBK, 1,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  } else {
    tmS = tmZ;  // never loaded
  }
  GemmArgs a;
  a.M = static_cast<int>(M);
  a.D_in = static_cast<int>(D_in);
  a.D_out = static_cast<int>(D_out);
  a.group_size = group_size;
  a.has_s = s != nullptr;
  a.m_blocks = static_cast<int>((M + 2 * kStack * kSubRows - 1) / (2 * kStack * kSubRows));
  a.n_blocks = static_cast<int>((D_out + kPairN - 1) / kPairN);
  a.num_tiles = a.m_blocks * a.n_blocks;
  a.Y = static_cast<__nv_bfloat16*>(Y);
  a.status = status;
  const size_t smem = static_cast<size_t>(kSmemBytes) + 1024;
  e = cudaFuncSetAttribute(w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int pairs = max_pairs;
  if (pairs > a.num_tiles) pairs = a.num_tiles;
  if (pairs < 1) pairs = 1;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(pairs, smem, stream, attr);
  return cudaLaunchKernelEx(&cfg, w4a16_kernel, tmX, tmC, tmSc, tmZ, tmS, a);
}

// ---------------------------------------------------------------------------
// Decode-sized W4A16 product (M <= 4 rows of X).  A few rows of X make the
// product a stream over the codes: every code byte is read once and used for
// M rows, so the kernel must turn 4-bit codes into products at HBM speed.  It
// does so on the tensor cores through register-fed mma.sync (m16n8k16, bf16
// in, fp32 accumulate), which keeps the codes in registers: a tcgen05 tile
// (M >= 64) would be mostly padding here and would force the unpacked
// weights through shared memory.
//
// Unpacking.  A 32-bit word of one byte row holds the codes of 4 columns
// c .. c+3 for input rows 2j (low nibbles) and 2j+1 (high nibbles).  One
// masked OR (w >> 4s) & 0x000F000F | 0x43004300 turns it into the bf16 pair
// (128 + q[row][c + s'], 128 + q[row][c + s' + 2]) -- 128 + q is exact in
// bf16 -- so 8 codes cost 3 shifts and 4 logic operations.  The pair holds
// two columns of one row, so the MMA's reduction index runs over
// (row, parity e in {0, 1}) with column c + 2e, and B carries x' in the slot
// of its own parity and zero in the other:
//   A (16 x 16): row g <-> column base c_g (rows g + 8: c_g + 1),
//                k = 2t + e <-> (input row of k pair t, column offset 2e);
//   B (16 x 8):  n = 4e' + 2m + h <-> (parity e', row m of X, x'_hi or
//                x'_lo), with x'_hi = bf16(x'), x'_lo = bf16(x' - x'_hi) of
//                x' = x / s, so the bf16 products lose nothing beyond 2^-16
//                of x'; B[(row, e)][n] = x'_h[row][m] if e = e' else 0;
//   D (16 x 8):  D[g][n] = sum over the rows of (128 + q[row][c_g + 2e'])
//                x'_h[row][m].
// Per group, with xs = sum of x'_hi + x'_lo over the group's rows (fp32,
// fixed order): y += sc (D_hi + D_lo - (z + 128) xs) = sc sum_j x'_j (q_j - z)
// ("AWQ (Activation-aware Weight Quantization)", 量化数学基础 step 3:
// Dequant = (q - z) s).  Rows 2 and 3 of X take a second n tile.
//
// A stage is 64 input rows x 1024 columns (32 KB of code bytes, eight
// 128-column tensor copies with the 128-byte swizzle) plus the rows' B
// fragments and row sums (xprep_kernel writes them once per call) and the
// group row of fp16 scales and zeros.  Consumer warp w owns columns
// 64w .. 64w+63; a k group is the 4 byte rows 8b + 2t + par (t = 0..3) of
// one parity in a block b of 8, so the 8-byte loads of a warp meet no bank
// conflicts under the swizzle; lane (g, t) = (lane / 4, lane % 4) loads
// columns 8g .. 8g+7 of byte row 8b + 2t + par, two words for two MMA tiles.
// Stages are taken in column-block-major order; persistent CTAs own equal
// contiguous runs of stages.  Where a run leaves a column block the CTA's
// sums go to slot (CTA + column block) of the workspace (the pair grows
// along every run, so slots never collide); the last CTA to finish a column
// block (a ticket counter per block) adds its segments top to bottom as
// fixed fp32 pairwise trees of 8 and writes Y in bf16.
namespace {

constexpr int kDqCols = 1024;                              // columns per stage
constexpr int kDqBoxCols = 128;                            // per tensor copy (128-byte swizzle)
constexpr int kDqWarpCols = 64;                            // per consumer warp
constexpr int kDqRows = 64;                                // input rows per stage
constexpr int kDqByteRows = kDqRows / 2;
constexpr int kDqKGroups = kDqByteRows / 4;                // 8 k groups of 4 byte rows
constexpr int kDqConsumers = kDqCols / kDqWarpCols;        // 16
constexpr int kDqThreads = (kDqConsumers + 1) * 32;
constexpr int kDqStages = 5;
constexpr int kDqCtasPerSm = 1;
constexpr int kDqNTiles = 2;                               // n tiles: rows 0-1 and 2-3 of X
constexpr int kDqCodeBytes = kDqByteRows * kDqCols;        // 32 KB
constexpr int kDqBoxBytes = kDqByteRows * kDqBoxCols;      // 4 KB, 1024-byte aligned
constexpr int kDqFragBytes = kDqKGroups * kDqNTiles * 32 * 8;  // B fragments of 64 rows
constexpr int kDqChunkBytes = kDqFragBytes + 16;           // + xs of the 64 rows for 4 rows of X
constexpr int kDqSideBytes = kDqCols * 2;                  // one group row of fp16
constexpr int kDqSideBox = 256;                            // fp16 columns per side copy
constexpr int kDqOffFrag = kDqCodeBytes;
constexpr int kDqOffSc = (kDqOffFrag + kDqChunkBytes + 127) / 128 * 128;
constexpr int kDqOffZ = kDqOffSc + kDqSideBytes;
constexpr int kDqStageTx = kDqCodeBytes + kDqChunkBytes + 2 * kDqSideBytes;
constexpr int kDqStageStride = (kDqOffZ + kDqSideBytes + 1023) / 1024 * 1024;
constexpr int kDqSmem = kDqStages * kDqStageStride + 1024;  // + alignment slack
constexpr int64_t kDqMaxCtas = 1024;                       // bound of the grid (workspace sizing)
constexpr uint32_t kDqBias = 0x43004300u;                  // bf16 pair (128, 128)
static_assert(kDqSmem <= 227 * 1024 && kDqCtasPerSm * (kDqSmem + 1024) <= 228 * 1024, "shared memory per SM");
static_assert(kDqChunkBytes % 16 == 0 && kDqOffSc % 128 == 0 && kDqOffZ % 128 == 0, "copy alignment");
static_assert(kDqOffFrag + kDqChunkBytes <= kDqOffSc && kDqOffZ + kDqSideBytes <= kDqStageStride,
              "every region a stage is read at lies inside the stage");

// (x & 0x000F000F) | bias in one logic operation (bias kept in a register).
__device__ __forceinline__ uint32_t code_pair(uint32_t x, uint32_t bias) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(d) : "r"(x), "r"(bias));
  return d;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 lds_u32x2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t bf16_bits(__nv_bfloat16 h) { return *reinterpret_cast<const uint16_t*>(&h); }

// x' = x / s (x when s is null), zero for rows of X past M.
__device__ __forceinline__ float xprime(const __nv_bfloat16* X, int M, int64_t D_in, const float* s, int m,
                                        int64_t row) {
  if (m >= M) return 0.f;
  const float v = __bfloat162float(X[static_cast<int64_t>(m) * D_in + row]);
  return s ? __fdiv_rn(v, s[row]) : v;
}
__device__ __forceinline__ void split_hi_lo(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// One CTA per 64-row chunk: the B fragments of its 8 k groups and 2 n tiles
// in the order the MMA reads them, and, per row of X, xs = sum of x'_hi +
// x'_lo over the 64 rows in row order.  CTA 0 also zeroes the workspace
// header (status word) and the ticket counters of the product that follows,
// which may start before this grid ends (programmatic dependent launch) and
// reads none of this before it waits for it.
constexpr int kXprepThreads = 4 * kDqRows;
__global__ void __launch_bounds__(kXprepThreads) xprep_kernel(const __nv_bfloat16* __restrict__ X, int M,
                                                              int64_t D_in, const float* __restrict__ s,
                                                              uint8_t* __restrict__ xf, uint32_t* __restrict__ header,
                                                              unsigned int* __restrict__ tickets, int64_t ntickets) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t ch = blockIdx.x;
  uint8_t* dst = xf + ch * kDqChunkBytes;
  const int tid = threadIdx.x, lane = tid & 31, kg = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int e = g >> 2, h = g & 1;
  const int blk = kg >> 1, par = kg & 1;
  const int64_t r_lo = ch * kDqRows + 16 * blk + 4 * t + 2 * par;  // byte row 8 blk + 2t + par, low nibble
  if (ch == 0) {
    if (tid < 64) header[tid] = 0u;
    for (int64_t i = tid; i < ntickets; i += kXprepThreads) tickets[i] = 0u;
  }
#pragma unroll
  for (int nt = 0; nt < kDqNTiles; ++nt) {
    const int m = 2 * nt + ((g >> 1) & 1);
    uint32_t b[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      __nv_bfloat16 hi, lo;
      split_hi_lo(xprime(X, M, D_in, s, m, r_lo + q), hi, lo);
      const uint32_t v = bf16_bits(h ? lo : hi);
      b[q] = e ? (v << 16) : v;  // the slot of parity e; the other parity's slot is zero
    }
    reinterpret_cast<uint2*>(dst)[(kg * kDqNTiles + nt) * 32 + lane] = make_uint2(b[0], b[1]);
  }
  // xs: thread (m, r) of the first 256 takes row r; a butterfly over the warp's
  // 32 rows, then the two warps of each row of X in order
  __shared__ float wsum[8];
  {
    __nv_bfloat16 hi, lo;
    split_hi_lo(xprime(X, M, D_in, s, tid / kDqRows, ch * kDqRows + tid % kDqRows), hi, lo);
    float v = __bfloat162float(hi) + __bfloat162float(lo);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) wsum[tid >> 5] = v;
  }
  __syncthreads();
  if (tid < 4) reinterpret_cast<float*>(dst + kDqFragBytes)[tid] = wsum[2 * tid] + wsum[2 * tid + 1];
}

// The CTA whose run holds stage b: the largest c with floor(c B / ctas) <= b.
__device__ __forceinline__ int64_t dq_cta_of(int64_t b, int64_t B, int64_t ctas) { return ((b + 1) * ctas - 1) / B; }

template <int NT>
__global__ void __launch_bounds__(kDqThreads, kDqCtasPerSm)
    w4a16_decode_kernel(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmSc,
                        const __grid_constant__ CUtensorMap tmZ, const uint8_t* __restrict__ xf, int M,
                        int64_t D_in, int64_t D_out, int group_size, uint32_t bias, float* __restrict__ partial,
                        unsigned int* __restrict__ tickets, __nv_bfloat16* __restrict__ Y, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kDqStages];
  __shared__ __align__(8) uint64_t empty_bar[kDqStages];
  __shared__ int abort_sh;
  __shared__ bool last;
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nch = D_in / kDqRows;                       // 64-row chunks per column block
  const int64_t ncb = (D_out + kDqCols - 1) / kDqCols;
  const int64_t B = nch * ncb, ctas = gridDim.x;
  const int64_t b_begin = static_cast<int64_t>(blockIdx.x) * B / ctas;
  const int64_t b_end = (static_cast<int64_t>(blockIdx.x) + 1) * B / ctas;
  const int64_t cpg = group_size / kDqRows;                 // chunks per group
  if (threadIdx.x == 0) {
    for (int st = 0; st < kDqStages; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], kDqConsumers);
    }
    abort_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDqConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmC);
      prefetch_tmap(&tmSc);
      prefetch_tmap(&tmZ);
      auto issue_codes_sides = [&](int st, int64_t cb, int64_t ch) {
        uint8_t* stage = smem + st * kDqStageStride;
        mbar_arrive_expect_tx(&full_bar[st], kDqStageTx);
        const int32_t c0 = static_cast<int32_t>(cb * kDqCols);
#pragma unroll
        for (int q = 0; q < kDqCols / kDqBoxCols; ++q)
          tma_load_2d(stage + q * kDqBoxBytes, &tmC, &full_bar[st], c0 + q * kDqBoxCols,
                      static_cast<int32_t>(ch * kDqByteRows));
        const int32_t g = static_cast<int32_t>(ch / cpg);
#pragma unroll
        for (int q = 0; q < kDqCols / kDqSideBox; ++q) {
          tma_load_2d(stage + kDqOffSc + q * kDqSideBox * 2, &tmSc, &full_bar[st], c0 + q * kDqSideBox, g);
          tma_load_2d(stage + kDqOffZ + q * kDqSideBox * 2, &tmZ, &full_bar[st], c0 + q * kDqSideBox, g);
        }
      };
      auto issue_frag = [&](int st, int64_t ch) {
        bulk_copy_g2s(smem + st * kDqStageStride + kDqOffFrag, xf + ch * kDqChunkBytes, kDqChunkBytes, &full_bar[st]);
      };
      // The first stages' codes and scales do not depend on the x' preparation
      // that may still run: issue them, then wait for it, then its fragments.
      const int pre = static_cast<int>(b_end - b_begin < kDqStages ? b_end - b_begin : kDqStages);
      {
        int64_t cb = b_begin / nch, ch = b_begin % nch;
        for (int j = 0; j < pre; ++j) {
          issue_codes_sides(j, cb, ch);
          if (++ch == nch) {
            ch = 0;
            ++cb;
          }
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        ch = b_begin % nch;
        for (int j = 0; j < pre; ++j) {
          issue_frag(j, ch);
          if (++ch == nch) ch = 0;
        }
      }
      int64_t cb = (b_begin + pre) / nch, ch = (b_begin + pre) % nch;
      int it = pre;
      bool ok = true;
      for (int64_t b = b_begin + pre; b < b_end; ++b, ++it) {
        const int st = it % kDqStages;
        if (!mbar_wait(&empty_bar[st], ((it / kDqStages) + 1) & 1, status, abort_flag)) {
          ok = false;
          break;
        }
        issue_codes_sides(st, cb, ch);
        issue_frag(st, ch);
        if (++ch == nch) {
          ch = 0;
          ++cb;
        }
      }
      // after an abort, the copies still in flight land before the CTA exits
      if (!ok || *abort_flag)
        for (int j = it - kDqStages < 0 ? 0 : it - kDqStages; j < it; ++j)
          mbar_wait(&full_bar[j % kDqStages], (j / kDqStages) & 1, nullptr, nullptr, kCopyDrainNs);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the tickets are zeroed by the preparation grid
  const int g = lane >> 2, t = lane & 3;
  // this lane's output: rows m = 2nt + (t & 1) of X, columns 8g + 4u + 2(t >> 1) + {0, 1} (u = 0, 1)
  const int ccol = warp * kDqWarpCols + 8 * g + 2 * (t >> 1);
  int64_t cb = b_begin / nch, ch = b_begin % nch;
  int64_t gch = ch % cpg;  // chunk index within its group
  int st = 0;
  uint32_t phase = 0;
  bool ok = true;    // false once a wait gave up; the warps leave together
  float y[NT][4];    // [n tile][2u + column offset]
  float d[NT][2][4];  // the group's MMA sums per n tile and MMA tile u
  float xs[NT];      // the group's row sums of x'_hi + x'_lo, rows 2nt + (t & 1) of X
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    xs[n] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) y[n][j] = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) d[n][u][k] = 0.f;
  }
  // Shared-memory byte offsets within a stage.  The warp's 64 columns are half
  // (warp & 1) of tensor copy warp / 2; the lane's 8 bytes of byte row p sit in
  // the 16-byte unit ((warp & 1) * 4 + g / 2) ^ (p & 7).  A k group of parity par
  // in block b of 8 byte rows takes byte row 8b + 2t + par, whose p & 7 = 2t + par.
  const uint32_t unit = (warp & 1) * 4 + (g >> 1);
  const uint32_t code_off = (warp >> 1) * kDqBoxBytes + (g & 1) * 8;
  const uint32_t row_off0 = code_off + (2 * t) * 128 + ((unit ^ (2 * t)) << 4);
  const uint32_t row_off1 = code_off + (2 * t + 1) * 128 + ((unit ^ (2 * t + 1)) << 4);
  const uint32_t frag_off = kDqOffFrag + lane * 8;
  const uint32_t smem_base = smem_u32(smem);
  for (int64_t b = b_begin; b < b_end; ++b) {
    if (ok && !mbar_wait(&full_bar[st], phase, status, abort_flag)) ok = false;
    const bool seg_end = ch == nch - 1 || b == b_end - 1;
    if (ok) {
      const uint32_t sa = smem_base + st * kDqStageStride;
#pragma unroll
      for (int kg = 0; kg < kDqKGroups; ++kg) {
        // byte row 8 (kg / 2) + 2t + (kg & 1): input rows 2p (low nibbles) and 2p + 1
        const uint2 cwd = lds_u32x2(sa + ((kg & 1) ? row_off1 : row_off0) + (kg >> 1) * 1024);
        const uint32_t w[2] = {cwd.x, cwd.y};
        uint2 bf[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) bf[n] = lds_u32x2(sa + frag_off + (kg * kDqNTiles + n) * 256);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t a0 = code_pair(w[u], bias), a1 = code_pair(w[u] >> 8, bias);
          const uint32_t a2 = code_pair(w[u] >> 4, bias), a3 = code_pair(w[u] >> 12, bias);
#pragma unroll
          for (int n = 0; n < NT; ++n) mma_bf16_16816(d[n][u], a0, a1, a2, a3, bf[n].x, bf[n].y);
        }
      }
      const uint8_t* stage = smem + st * kDqStageStride;
      const float* xsum = reinterpret_cast<const float*>(stage + kDqOffFrag + kDqFragBytes);
#pragma unroll
      for (int n = 0; n < NT; ++n) xs[n] += xsum[2 * n + (t & 1)];
      if (gch == cpg - 1 || seg_end) {
        // the group (or the run's part of it) ends: y += sc (D_hi + D_lo - (z + 128) xs)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(stage + kDqOffSc + (ccol + 4 * u) * 2));
          const float2 z = __half22float2(*reinterpret_cast<const __half2*>(stage + kDqOffZ + (ccol + 4 * u) * 2));
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            y[n][2 * u] = fmaf(sc.x, fmaf(-(z.x + 128.f), xs[n], d[n][u][0] + d[n][u][1]), y[n][2 * u]);
            y[n][2 * u + 1] = fmaf(sc.y, fmaf(-(z.y + 128.f), xs[n], d[n][u][2] + d[n][u][3]), y[n][2 * u + 1]);
#pragma unroll
            for (int k = 0; k < 4; ++k) d[n][u][k] = 0.f;
          }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) xs[n] = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);  // the warp is done with the stage
    }
    if (++st == kDqStages) {
      st = 0;
      phase ^= 1u;
    }
    if (++gch == cpg) gch = 0;
    if (seg_end) {
      if (named_bar_or(1, kDqConsumers * 32, !ok)) return;  // all consumer warps, after an abort
      const int64_t slot = blockIdx.x + cb;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int m = 2 * n + (t & 1);
        if (m < M) {
          float* dst = partial + (slot * M + m) * kDqCols + ccol;
          *reinterpret_cast<float2*>(dst) = make_float2(y[n][0], y[n][1]);
          *reinterpret_cast<float2*>(dst + 4) = make_float2(y[n][2], y[n][3]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) y[n][j] = 0.f;
      }
      __threadfence();
      named_bar_sync(1, kDqConsumers * 32);
      const int64_t c_first = dq_cta_of(cb * nch, B, ctas), c_last = dq_cta_of((cb + 1) * nch - 1, B, ctas);
      if (threadIdx.x == 0) last = atomicAdd(&tickets[cb], 1u) == static_cast<unsigned>(c_last - c_first);
      named_bar_sync(1, kDqConsumers * 32);
      if (last) {
        __threadfence();
        const int64_t nseg = c_last - c_first + 1;
        // thread k sums columns k and k + 512 of the block for every row of X
        const int k0 = threadIdx.x;
        for (int m = 0; m < M; ++m) {
#pragma unroll 1
          for (int q = 0; q < kDqCols / (kDqConsumers * 32); ++q) {
            const int64_t col = cb * kDqCols + q * kDqConsumers * 32 + k0;
            const float* src = partial + ((c_first + cb) * M + m) * kDqCols + q * kDqConsumers * 32 + k0;
            float v = 0.f;
            for (int64_t b0 = 0; b0 < nseg; b0 += 8) {
              // the segments in batches of 8, each a fixed pairwise fp32 tree, the batches in order
              float pv[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) pv[k] = b0 + k < nseg ? __ldcg(src + (b0 + k) * M * kDqCols) : 0.f;
#pragma unroll
              for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                for (int k = 0; k < w; ++k) pv[k] += pv[k + w];
              v += pv[0];
            }
            if (col < D_out) Y[static_cast<int64_t>(m) * D_out + col] = __float2bfloat16_rn(v);
          }
        }
        if (threadIdx.x == 0) tickets[cb] = 0u;  // ready for the next call
      }
      named_bar_sync(1, kDqConsumers * 32);  // `last` is rewritten at the next segment's end
    }
    if (++ch == nch) {
      ch = 0;
      gch = 0;
      ++cb;
    }
  }
}

}  // namespace

int64_t w4a16_decode_partial_floats(int64_t M, int64_t D_in, int64_t D_out) {
  (void)D_in;
  return (kDqMaxCtas + (D_out + kDqCols - 1) / kDqCols) * M * kDqCols;
}
int64_t w4a16_decode_tickets(int64_t D_out) { return (D_out + kDqCols - 1) / kDqCols; }
int64_t w4a16_decode_xprep_bytes(int64_t D_in) { return (D_in / kDqRows) * kDqChunkBytes; }

cudaError_t launch_w4a16_decode(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, int64_t M, int64_t D_in,
                                int64_t D_out, const uint8_t* qweight, const void* scales, const void* zeros,
                                const float* s, int group_size, void* Y, float* partial, unsigned int* tickets,
                                uint8_t* xf, uint32_t* status, cudaStream_t stream) {
  if (M < 1 || M > kW4a16DecodeMaxRows || D_in % kDqRows != 0 || group_size % kDqRows != 0)
    return cudaErrorInvalidValue;
  CUtensorMap tmC, tmSc, tmZ;
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D_out), static_cast<cuuint64_t>(D_in / 2)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D_out)};
    const cuuint32_t box[2] = {kDqBoxCols, kDqByteRows};
    if (encode(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(qweight), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D_out), static_cast<cuuint64_t>(D_in / group_size)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D_out) * 2};
    const cuuint32_t box[2] = {kDqSideBox, 1};
    if (encode(&tmSc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(scales), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&tmZ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(zeros), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // the CTAs that fit on the device, queried once per device (both kernels have the same footprint)
  static std::atomic<int> resident[64];
  auto kern = M <= 2 ? w4a16_decode_kernel<1> : w4a16_decode_kernel<2>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int fit = resident[dev].load(std::memory_order_acquire);
  if (fit == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDqThreads, kDqSmem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    fit = sms * per_sm;
    resident[dev].store(fit, std::memory_order_release);
  }
  const int64_t nch = D_in / kDqRows;
  const int64_t ncb = (D_out + kDqCols - 1) / kDqCols;
  xprep_kernel<<<static_cast<unsigned>(nch), kXprepThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(X), static_cast<int>(M), D_in, s, xf, status, tickets, ncb);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the product starts while the preparation runs (its codes do not depend on it)
  const int64_t ctas = std::min<int64_t>(std::min<int64_t>(fit, kDqMaxCtas), nch * ncb);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kDqThreads);
  cfg.dynamicSmemBytes = kDqSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tmC, tmSc, tmZ, static_cast<const uint8_t*>(xf), static_cast<int>(M), D_in,
                         D_out, group_size, kDqBias, partial, tickets, static_cast<__nv_bfloat16*>(Y), status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace awqdev
