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
// Decode-sized W4A16 product (M <= 4 rows of X): the codes are read once and
// the work is a handful of FMAs per weight, so CUDA cores keep up with HBM.
// A CTA owns 256 columns x 256 input rows; warp w takes rows 32w .. 32w+31
// (inside one group for every group size), lane l columns 8l .. 8l+7, one
// 8-byte code load per byte row.  x' = x / s of the CTA's rows sits in shared
// memory.  Per group the dequantisation is factored out of the sum:
//   sum_j x'_j (q_j - z) sc = sc (sum_j x'_j q_j - z sum_j x'_j),
// so a weight costs a nibble unpack and one FMA per row of X.  The 8 warps'
// sums are added in warp order, the CTA's partial goes to the workspace, and
// the last CTA of a column block (ticket) adds the row blocks in a fixed
// order (fp32 pairwise trees of 16, then in order) and writes Y in bf16.
namespace {

constexpr int kDecCols = 256;       // columns per CTA (32 lanes x 8)
constexpr int kDecRows = 256;       // input rows per CTA (8 warps x 32)
constexpr int kDecThreads = 256;

template <int MT>
__global__ void __launch_bounds__(kDecThreads)
    w4a16_decode_kernel(const __nv_bfloat16* __restrict__ X, int M, int64_t D_in, int64_t D_out,
                        const uint8_t* __restrict__ qweight, const __half* __restrict__ scales,
                        const __half* __restrict__ zeros, const float* __restrict__ s, int group_size,
                        float* __restrict__ partial, unsigned int* __restrict__ tickets, __nv_bfloat16* __restrict__ Y) {
  __shared__ float xs[MT][kDecRows];                  // x' = x / s of the CTA's rows
  __shared__ float red[kDecThreads / 64][MT][kDecCols];  // warps w and w + 4 add into slot w
  __shared__ bool last;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kDecCols;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kDecRows;
  const int rows = static_cast<int>(min(static_cast<int64_t>(kDecRows), D_in - r0));  // a multiple of 64
  for (int i = t; i < MT * kDecRows; i += kDecThreads) {
    const int m = i / kDecRows, r = i % kDecRows;
    float v = 0.f;
    if (m < M && r < rows) {
      v = __bfloat162float(X[static_cast<int64_t>(m) * D_in + r0 + r]);
      if (s) v = __fdiv_rn(v, s[r0 + r]);
    }
    xs[m][r] = v;
  }
  __syncthreads();

  const int64_t n = n0 + lane * 8;
  float acc[MT][8];  // sum_j x'_j q_j of the warp's rows, then its share of Y
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[m][c] = 0.f;
  const int wr = warp * 32;  // the warp's first row within the CTA
  if (wr < rows && n < D_out) {
    const uint8_t* qb = qweight + ((r0 + wr) / 2) * D_out + n;
    // the warp's 16 byte rows in batches whose loads are all in flight: one
    // batch of 16 for one or two rows of X, two of 8 when the accumulators
    // need the registers
    constexpr int kBatch = MT <= 2 ? 16 : 8;
#pragma unroll
    for (int h = 0; h < 16 / kBatch; ++h) {
      uint2 cb[kBatch];
#pragma unroll
      for (int p = 0; p < kBatch; ++p) cb[p] = *reinterpret_cast<const uint2*>(qb + (kBatch * h + p) * D_out);
#pragma unroll
      for (int p = 0; p < kBatch; ++p) {
#pragma unroll
        for (int odd = 0; odd < 2; ++odd) {
          float t0[4], t1[4];
          nibbles_to_f32(odd ? (cb[p].x >> 4) & 0x0F0F0F0Fu : cb[p].x & 0x0F0F0F0Fu, t0);
          nibbles_to_f32(odd ? (cb[p].y >> 4) & 0x0F0F0F0Fu : cb[p].y & 0x0F0F0F0Fu, t1);
          float qc[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            qc[k] = t0[k] - 8388608.0f;  // the code, exact
            qc[4 + k] = t1[k] - 8388608.0f;
          }
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const float x = xs[m][wr + 2 * (kBatch * h + p) + odd];
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[m][c] = fmaf(x, qc[c], acc[m][c]);
          }
        }
      }
    }
    // the warp's rows lie in one group: scale and zero of its 8 columns
    const int64_t g = (r0 + wr) / group_size;
    const uint4 hs = *reinterpret_cast<const uint4*>(scales + g * D_out + n);
    const uint4 hz = *reinterpret_cast<const uint4*>(zeros + g * D_out + n);
    const uint32_t us[4] = {hs.x, hs.y, hs.z, hs.w};
    const uint32_t uz[4] = {hz.x, hz.y, hz.z, hz.w};
    float sc[8], zc[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&us[k]));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&uz[k]));
      sc[2 * k] = a.x;
      sc[2 * k + 1] = a.y;
      zc[2 * k] = b.x;
      zc[2 * k + 1] = b.y;
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float xsum = 0.f;
#pragma unroll 8
      for (int r = 0; r < 32; ++r) xsum += xs[m][wr + r];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[m][c] = sc[c] * fmaf(-zc[c], xsum, acc[m][c]);
    }
  }
  // the 8 warps' shares in a fixed order: (w0 + w4) + (w1 + w5) + (w2 + w6) + (w3 + w7)
  if (warp < 4) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float4* dst = reinterpret_cast<float4*>(&red[warp][m][lane * 8]);
      dst[0] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      dst[1] = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
    }
  }
  __syncthreads();
  if (warp >= 4) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float4* dst = reinterpret_cast<float4*>(&red[warp - 4][m][lane * 8]);
      const float4 a = dst[0], b = dst[1];
      dst[0] = make_float4(a.x + acc[m][0], a.y + acc[m][1], a.z + acc[m][2], a.w + acc[m][3]);
      dst[1] = make_float4(b.x + acc[m][4], b.y + acc[m][5], b.z + acc[m][6], b.w + acc[m][7]);
    }
  }
  __syncthreads();
  const int64_t rb_count = gridDim.y;
  for (int i = t; i < MT * kDecCols; i += kDecThreads) {
    const int m = i / kDecCols, c = i % kDecCols;
    if (m < M && n0 + c < D_out) {
      const float v = (red[0][m][c] + red[1][m][c]) + (red[2][m][c] + red[3][m][c]);
      partial[(static_cast<int64_t>(blockIdx.y) * M + m) * D_out + n0 + c] = v;
    }
  }
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&tickets[blockIdx.x], 1u) == static_cast<unsigned>(rb_count) - 1u;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = t; i < MT * kDecCols; i += kDecThreads) {
    const int m = i / kDecCols, c = i % kDecCols;
    if (m < M && n0 + c < D_out) {
      // 16 row blocks' loads in flight, each batch as a fixed pairwise fp32
      // tree, the batches in order (fp64 adds are slow on this part)
      float v = 0.f;
      for (int64_t b0 = 0; b0 < rb_count; b0 += 16) {
        float pv[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          pv[k] = b0 + k < rb_count ? partial[((b0 + k) * M + m) * D_out + n0 + c] : 0.f;
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int k = 0; k < w; ++k) pv[k] += pv[k + w];
        v += pv[0];
      }
      Y[static_cast<int64_t>(m) * D_out + n0 + c] = __float2bfloat16_rn(v);
    }
  }
  if (t == 0) tickets[blockIdx.x] = 0u;  // ready for the next call
}

}  // namespace

int64_t w4a16_decode_partial_floats(int64_t M, int64_t D_in, int64_t D_out) {
  return ((D_in + kDecRows - 1) / kDecRows) * M * D_out;
}
int64_t w4a16_decode_tickets(int64_t D_out) { return (D_out + kDecCols - 1) / kDecCols; }

cudaError_t launch_w4a16_decode(const void* X, int64_t M, int64_t D_in, int64_t D_out, const uint8_t* qweight,
                                const void* scales, const void* zeros, const float* s, int group_size, void* Y,
                                float* partial, unsigned int* tickets, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((D_out + kDecCols - 1) / kDecCols),
                  static_cast<unsigned>((D_in + kDecRows - 1) / kDecRows));
  const auto* Xb = static_cast<const __nv_bfloat16*>(X);
  const auto* sc = static_cast<const __half*>(scales);
  const auto* zr = static_cast<const __half*>(zeros);
  auto* Yb = static_cast<__nv_bfloat16*>(Y);
  const int m = static_cast<int>(M);
  if (M <= 1)
    w4a16_decode_kernel<1><<<grid, kDecThreads, 0, stream>>>(Xb, m, D_in, D_out, qweight, sc, zr, s, group_size,
                                                             partial, tickets, Yb);
  else if (M <= 2)
    w4a16_decode_kernel<2><<<grid, kDecThreads, 0, stream>>>(Xb, m, D_in, D_out, qweight, sc, zr, s, group_size,
                                                             partial, tickets, Yb);
  else
    w4a16_decode_kernel<4><<<grid, kDecThreads, 0, stream>>>(Xb, m, D_in, D_out, qweight, sc, zr, s, group_size,
                                                             partial, tickets, Yb);
  return cudaGetLastError();
}

}  // namespace awqdev
