// Fused candidate search on a tcgen05 CTA pair (sm_103a).
//
// For candidate k the search needs the output error of the quantised layer,
//   E_k = X * S_k^-1 W'hat_k - X * W = X * D_k,  D_k = S_k^-1 W'hat_k - W,
// and only the per-column sums of squares of E_k ("AWQ (Activation-aware
// Weight Quantization)", 缩放因子优化的完整流程 steps 3-4: scale, quantise
// per group, dequantise, L = ||X S^-1 W'hat - X W||^2).  D_k is never stored:
// producer warps build each bf16 tile of it in registers from W, the scale
// row s_k and the per-group step / zero, and write it straight into the
// shared-memory operand layout of the tensor cores.
//
// Work unit: (candidate k, 512 rows of X, 256 columns of W).  Two CTAs of a
// cluster form a tcgen05 pair: each holds two stacked 128-row subtiles of X
// (rows m0 + 256*s + 128*rank) and produces half (128 columns) of the D_k
// tile; the even CTA issues M256 x N256 x K16 MMAs that read A from both CTAs
// and B from both halves, accumulating in fp32 TMEM (2 subtiles x 256
// columns = all 512 TMEM columns of each CTA).  Every produced element of D_k
// feeds 512 rows of MMA work, which keeps the producer's CUDA-core cost well
// under the tensor-core time of the same K step.
//
// The W tile of a K step is loaded by TMA with 128-byte swizzle straight into
// the B operand slot, which is the tensor cores' N-major layout; each
// producer thread reads its 16-byte chunks there and overwrites them in
// place with the same chunks of D.  X (A operand, 4 stages) and W/D (B
// operand, 5 stages) have separate rings; the small per-step inputs of the
// producers (s and 1/s of the 64 rows, step / zero of the group) ride in a
// side slot of the B ring.
//
// Roles (640 threads per CTA):
//   warp 0      TMA: X subtiles (K-major, 128-byte swizzle) per K step; the
//               completion is counted on the even CTA's barrier
//   warp 1      TMEM allocation; in the even CTA the single-thread MMA issuer
//   warp 2      TMA: W tile into the B slot and the side inputs, per K step
//   warps 4-11  epilogue: TMEM -> registers, square, column sums over the
//               CTA's 256 rows (fixed order), one fp32 partial per column
//   warps 12-19 producers: two groups of 4 warps on alternate K steps
//               (128 threads, 8 columns x 8 rows each per step)
// The kernel is persistent: each pair walks the work units with a stride of
// the number of pairs.  Every mbarrier wait is bounded; a timeout records
// AWQ_ERR_TIMEOUT and every role leaves its loop.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {
namespace {

constexpr int kBK = 64;                        // K (input rows of W) per step
constexpr int kSubRows = 128;                  // X rows of one subtile in one CTA
constexpr int kStack = 2;                      // stacked subtiles per CTA
constexpr int kPairN = 256;                    // columns of W per work unit
constexpr int kHalfN = kPairN / 2;             // columns produced by one CTA
constexpr int kAStages = 4;                    // X ring
constexpr int kBStages = 5;                    // W -> D ring
constexpr int kASubBytes = kSubRows * kBK * 2;  // 16 KB
constexpr int kABytes = kStack * kASubBytes;    // 32 KB
constexpr int kBBytes = kBK * kHalfN * 2;       // 16 KB: 64 K x 128 N bf16, N-major, 128B swizzle
constexpr int kSBytes = kBK * 4;                // s slice (and 1/s slice)
constexpr int kQBytes = (kHalfN / kQChunkCols) * kQChunkFloats * 4;  // step / zero chunks of 128 columns
constexpr int kSideTx = 2 * kSBytes + kQBytes;
constexpr int kSideStride = (kSideTx + 127) / 128 * 128;  // TMA destinations stay 128-byte aligned
constexpr int kOffB = kAStages * kABytes;
constexpr int kOffSide = kOffB + kBStages * kBBytes;
constexpr int kSmemBytes = kOffSide + kBStages * kSideStride;
constexpr int kTmemCols = 512;
constexpr int kThreads = 640;
constexpr int kEpiWarp0 = 4, kEpiWarps = 8;
constexpr int kProdWarp0 = 12, kProdWarps = 8;
constexpr int kGroupWarps = 4;                   // producer warps per K step (two groups alternate)
static_assert(kProdWarps == 2 * kGroupWarps, "two producer groups");
constexpr int kBFullCount = 2 * kGroupWarps;     // one producer group of each CTA
constexpr int kAccEmptyCount = 2 * kEpiWarps;
constexpr int kHeadSteps = 3;                    // K steps a tile starts on subtile 0 alone
static_assert(kHeadSteps <= kAStages && kHeadSteps <= kBStages, "the held head steps fit in both rings");

static_assert(kSmemBytes + 1024 + 4608 <= 227 * 1024, "shared memory (dynamic + alignment slack + static)");

struct FusedArgs {
  int N, D_in, D_out, G, T, group_size;
  int m_blocks, n_blocks, num_tiles, m_tiles;
  int sb_m, sb_n;  // super-block: sb_m row bands x sb_n column blocks (see decode_tile)
  float clamp_lo, clamp_hi;
  float* partial;  // [G][m_tiles][D_out]
  uint32_t* status;
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Sum v[0..31] across the 32 lanes so that lane l ends with sum_lanes v[l].
__device__ __forceinline__ float transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
    }
  }
  return v[0];
}

// Four rows x 8 columns of the negated difference tile D = W - S^-1 W'hat:
//   w' = w s;  t = rint(w' / step) + zero, held as 1.5*2^23 + code;  clamp
//   to the code range;  d = (w' - (code - zero) step) / s.
// (D and -D give the same loss.)  CLAMP = false leaves out the clamps, for
// warps none of whose columns has a code outside the range in this group
// (the group-parameter table's per-chunk flag).  `w` points at the 16-byte chunk of row 0
// in the swizzled B slot; row i's chunk sits at w + i*128 with its 16-byte
// position XOR-ed by i (rows 4*half .. 4*half+3 of an 8-row swizzle atom).
// Each chunk of W is overwritten in place by the same chunk of D.
template <bool CLAMP>
__device__ __forceinline__ void produce4(uint8_t* w, int c8, int half, float4 s4, float4 r4,
                                         const float2 (&inv2)[4], const float2 (&zm2)[4],
                                         const float2 (&nzm2)[4], const float2 (&nstep2)[4], float lo, float hi) {
  const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
  const float rv[4] = {r4.x, r4.y, r4.z, r4.w};
  uint4 wv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    wv[i] = *reinterpret_cast<const uint4*>(w + i * 128 + ((c8 ^ (4 * half + i)) * 16));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t wu[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
    const float2 s2 = make_float2(sv[i], sv[i]);
    const float2 r2 = make_float2(rv[i], rv[i]);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 w2 = make_float2(bf16lo(wu[j]), bf16hi(wu[j]));
      const float2 wp = __fmul2_rn(w2, s2);
      float2 tq = __ffma2_rn(wp, inv2[j], zm2[j]);
      if (CLAMP) {
        tq.x = fminf(fmaxf(tq.x, lo), hi);
        tq.y = fminf(fmaxf(tq.y, lo), hi);
      }
      const float2 qz = __fadd2_rn(tq, nzm2[j]);
      const float2 ev = __ffma2_rn(qz, nstep2[j], wp);
      const float2 d = __fmul2_rn(ev, r2);
      o[j] = pack_bf16x2(d.x, d.y);
    }
    *reinterpret_cast<uint4*>(w + i * 128 + ((c8 ^ (4 * half + i)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

struct Tile {
  int k, m_blk, n_blk;
};
// Work units in an L2-sized order: candidate fastest, then the units of one
// super-block of sb_m row bands x sb_n column blocks (column block fastest),
// super-blocks column-major within a strip of sb_m bands, strips in order.
// A super-block's X rows, W columns and parameter rows stay in L2 while all
// candidates of all its units run, so W and the parameter table come from
// HBM once per strip instead of once per row band.
__device__ __forceinline__ Tile decode_tile(int t, const FusedArgs& p) {
  Tile r;
  r.k = t % p.G;
  const int u = t / p.G;
  const int strip = u / (p.sb_m * p.n_blocks);  // every earlier strip is full
  const int in_strip = u - strip * (p.sb_m * p.n_blocks);
  const int mb = min(p.sb_m, p.m_blocks - strip * p.sb_m);  // bands in this strip
  const int sbk = in_strip / (mb * p.sb_n);                 // every earlier super-block of the strip is full
  const int in_sb = in_strip - sbk * (mb * p.sb_n);
  const int nb = min(p.sb_n, p.n_blocks - sbk * p.sb_n);    // column blocks in this super-block
  r.m_blk = strip * p.sb_m + in_sb / nb;
  r.n_blk = sbk * p.sb_n + in_sb % nb;
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    search_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmR,
                        const __grid_constant__ CUtensorMap tmQ, FusedArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t afull_bar[kAStages];   // even CTA: X of both CTAs landed
  __shared__ __align__(8) uint64_t aempty_bar[kAStages];  // both CTAs: MMAs done with the X slot
  __shared__ __align__(8) uint64_t wfull_bar[kBStages];   // local: W tile and side inputs landed
  __shared__ __align__(8) uint64_t bfull_bar[kBStages];   // even CTA: D written by both CTAs
  __shared__ __align__(8) uint64_t bempty_bar[kBStages];  // both CTAs: MMAs done with the B slot
  __shared__ __align__(8) uint64_t acc_full_bar;          // both CTAs
  __shared__ __align__(8) uint64_t acc_empty_bar[kStack];  // even CTA: subtile s of the accumulator read out
  __shared__ __align__(8) uint64_t mma_drain_bar;          // even CTA: MMAs still running after an abort
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float red[4][kPairN];

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
      mbar_init(&wfull_bar[s], 1);
      mbar_init(&bfull_bar[s], kBFullCount);
      mbar_init(&bempty_bar[s], 1);
    }
    mbar_init(&acc_full_bar, 1);
    for (int sub = 0; sub < kStack; ++sub) mbar_init(&acc_empty_bar[sub], kAccEmptyCount);
    mbar_init(&mma_drain_bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32 * 2) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmS);
    prefetch_tmap(&tmR);
    prefetch_tmap(&tmQ);
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

  // shared::cluster addresses of the even CTA's barriers
  const uint32_t afull0 = mapa_shared(smem_u32(&afull_bar[0]), 0);
  const uint32_t bfull0 = mapa_shared(smem_u32(&bfull_bar[0]), 0);
  const uint32_t acc_empty0 = mapa_shared(smem_u32(&acc_empty_bar[0]), 0);

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
      // drain: the MMA commits of the last steps arrive on this CTA's empty
      // barriers; wait for them so that no arrival targets an exited CTA
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
      // M = 256 (pair), N = 256, bf16 x bf16 -> fp32, A K-major, B N-major
      constexpr uint32_t idesc = idesc_bf16_f32(256, kPairN, 0, 1);
      int it = 0, tc = 0;
      // Issue the MMAs of K step `it` for subtiles [sub0, sub1) of the accumulator.
      auto issue = [&](int it_, int kb, int sub0, int sub1) {
        const int sa = it_ % kAStages;
        const int sb = it_ % kBStages;
        const uint32_t a_addr = smem_u32(smem + sa * kABytes);
        const uint32_t b_addr = smem_u32(smem + kOffB + sb * kBBytes);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // B: N-major SW128; 64-column chunks 8 KB apart (LBO), 8-row K
          // groups 1024 B apart (SBO); a K step of 16 is two K groups.
          const uint64_t bd = sdesc_sw128(b_addr + kk * 2048, kBK * 128, 1024);
          for (int sub = sub0; sub < sub1; ++sub) {
            const uint64_t ad = sdesc_sw128(a_addr + sub * kASubBytes + kk * 32, 16, 1024);
            umma_bf16_pair(tmem + static_cast<uint32_t>(sub * kPairN), ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
      };
      auto inputs_ready = [&](int it_) {
        return mbar_wait_cluster(&afull_bar[it_ % kAStages], (it_ / kAStages) & 1, p.status, abort_flag) &&
               mbar_wait_cluster(&bfull_bar[it_ % kBStages], (it_ / kBStages) & 1, p.status, abort_flag);
      };
      auto release = [&](int it_) {
        umma_commit_pair_mc(&aempty_bar[it_ % kAStages], 0x3);
        umma_commit_pair_mc(&bempty_bar[it_ % kBStages], 0x3);
      };
      for (int t = pair; t < p.num_tiles; t += npairs, ++tc) {
        // The epilogue reads the previous tile's subtile 0 first and releases
        // it on its own barrier: the first kHeadSteps K steps of this tile
        // start on subtile 0 (holding their stages) while subtile 1 is still
        // being read out, which hides part of the drain between tiles.
        if (tc > 0 && !mbar_wait_cluster(&acc_empty_bar[0], (tc - 1) & 1, p.status, abort_flag)) break;
        tc_fence_after();
        const int head = KB < kHeadSteps ? KB : kHeadSteps;
        bool ok = true;
        for (int kb = 0; kb < head; ++kb) {
          if (!inputs_ready(it + kb)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue(it + kb, kb, 0, 1);
        }
        if (!ok) break;
        if (tc > 0 && !mbar_wait_cluster(&acc_empty_bar[1], (tc - 1) & 1, p.status, abort_flag)) break;
        tc_fence_after();
        for (int kb = 0; kb < head; ++kb) {
          issue(it + kb, kb, 1, kStack);
          release(it + kb);
        }
        it += head;
        for (int kb = head; kb < KB; ++kb, ++it) {
          if (!inputs_ready(it)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue(it, kb, 0, kStack);
          release(it);
        }
        if (!ok) break;
        umma_commit_pair_mc(&acc_full_bar, 0x3);
      }
      // the epilogues' last arrivals (some remote) land before the pair exits
      if (tc > 0 && !*abort_flag)
        for (int sub = 0; sub < kStack; ++sub)
          mbar_wait_cluster(&acc_empty_bar[sub], (tc - 1) & 1, p.status, abort_flag);
      if (*abort_flag) {
        // no MMA of the pair may still run when TMEM is freed: one more
        // commit arrives once every MMA issued so far is done
        umma_commit_pair_mc(&mma_drain_bar, 0x1);
        mbar_wait(&mma_drain_bar, 0, nullptr, nullptr, kCopyDrainNs);
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- W / side-input loader
    if (lane == 0) {
      int it = 0;
      for (int t = pair; t < p.num_tiles && !*abort_flag; t += npairs) {
        const Tile tl = decode_tile(t, p);
        const int n_base = tl.n_blk * kPairN + static_cast<int>(rank) * kHalfN;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % kBStages;
          const uint32_t ph = (it / kBStages) & 1;
          if (it >= kBStages && !mbar_wait_cluster(&bempty_bar[s], ph ^ 1, p.status, abort_flag)) break;
          uint8_t* bst = smem + kOffB + s * kBBytes;
          uint8_t* side = smem + kOffSide + s * kSideStride;
          mbar_arrive_expect_tx(&wfull_bar[s], kBBytes + kSideTx);
          tma_load_2d(bst, &tmW, &wfull_bar[s], n_base, kb * kBK);
          tma_load_2d(bst + kBBytes / 2, &tmW, &wfull_bar[s], n_base + 64, kb * kBK);
          tma_load_2d(side, &tmS, &wfull_bar[s], kb * kBK, tl.k);
          tma_load_2d(side + kSBytes, &tmR, &wfull_bar[s], kb * kBK, tl.k);
          tma_load_3d(side + 2 * kSBytes, &tmQ, &wfull_bar[s], 0, n_base / kQChunkCols,
                      tl.k * p.T + (kb * kBK) / p.group_size);
        }
        if (*abort_flag) break;
      }
      // drain: the MMA commits of the last steps arrive on this CTA's empty
      // barriers (which also implies every load landed)
      const int first = it - kBStages < 0 ? 0 : it - kBStages;
      for (int j = first; j < it; ++j)
        mbar_wait_cluster(&bempty_bar[j % kBStages], (j / kBStages) & 1, p.status, abort_flag);
      if (*abort_flag)  // after an abort: this CTA's own copies in flight land first
        for (int j = first; j < it; ++j)
          mbar_wait(&wfull_bar[j % kBStages], (j / kBStages) & 1, nullptr, nullptr, kCopyDrainNs);
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ---------------------------------------------------------- epilogue
    const int e = warp - kEpiWarp0;
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int ch = e >> 2;          // column half: [ch*128, ch*128 + 128)
    const int ecol = e * 32 + lane; // column of the final fixed-order sum
    int tc = 0;
    for (int t = pair; t < p.num_tiles; t += npairs, ++tc) {
      const Tile tl = decode_tile(t, p);
      // one warp polls the accumulator barrier; the other seven sleep in a
      // hardware barrier until it has seen the phase (no polling traffic for
      // the length of a tile), and all learn whether the wait succeeded
      bool ok = true;
      if (e == 0) ok = mbar_wait(&acc_full_bar, tc & 1, p.status, abort_flag);
      ok = !named_bar_or(2, kEpiWarps * 32, !ok);
      tc_fence_after();
      if (ok) {
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        // subtile 0, then subtile 1, each released as soon as this warp has
        // read it: per column, the sum of squares of each subtile's 128 rows
#pragma unroll 1
        for (int sub = 0; sub < kStack; ++sub) {
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            const int col = ch * 128 + cc * 32;
            float a[32];
            tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(sub * kPairN + col), a);
            if (cc == 3) {
              // every TMEM read of this subtile by this warp is complete
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_remote(acc_empty0 + static_cast<uint32_t>(sub) * 8u);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = a[i] * a[i];
            const float v = transpose_sum32(a, lane);
            if (sub == 0)
              red[q][col + lane] = v;
            else
              red[q][col + lane] += v;
          }
        }
      }
      if (named_bar_or(1, kEpiWarps * 32, !ok || *abort_flag)) break;
      {
        const float sum = ((red[0][ecol] + red[1][ecol]) + red[2][ecol]) + red[3][ecol];
        const int n = tl.n_blk * kPairN + ecol;
        const int mt = 2 * tl.m_blk + static_cast<int>(rank);
        if (n < p.D_out) p.partial[(static_cast<int64_t>(tl.k) * p.m_tiles + mt) * p.D_out + n] = sum;
      }
      named_bar_sync(1, kEpiWarps * 32);
    }
  } else if (warp >= kProdWarp0) {
    // ---------------------------------------------------------- producers
    // Two groups of 4 warps take alternate K steps, so that one group's
    // waits overlap the other's arithmetic.  Thread: 8 columns (chunk c) x 8
    // rows (8*rg .. 8*rg+7) of the 64 x 128 tile of its step.
    const int grp_id = (warp - kProdWarp0) / kGroupWarps;
    const int gt = threadIdx.x - (kProdWarp0 + grp_id * kGroupWarps) * 32;
    const int c = gt & 15;
    const int rg = gt >> 4;
    const int h = c >> 3;        // 64-column half of the CTA's 128 columns
    const int c8 = c & 7;        // 16-byte chunk inside a 128-byte row
    const float lo = p.clamp_lo, hi = p.clamp_hi;
    int it = 0;
    for (int t = pair; t < p.num_tiles && !*abort_flag; t += npairs) {
      int cached_group = -1;
      bool clampw = true;
      float2 inv2[4], zm2[4], nzm2[4], nstep2[4];
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        if ((it & 1) != grp_id) continue;
        const int s = it % kBStages;
        if (!mbar_wait(&wfull_bar[s], (it / kBStages) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* side = smem + kOffSide + s * kSideStride;
        const int grp = (kb * kBK) / p.group_size;
        if (grp != cached_group) {
          cached_group = grp;
          // chunk c: {1/step x8, 1.5*2^23 + zero x8, step x8, clamp flag, unused x3}
          const float4* qp = reinterpret_cast<const float4*>(side + 2 * kSBytes + c * (kQChunkFloats * 4));
          const float4 i0 = qp[0], i1 = qp[1], z0 = qp[2], z1 = qp[3], s0 = qp[4], s1 = qp[5];
          // one path per warp: the clamps stay unless no column of the warp needs them
          clampw = __any_sync(0xFFFFFFFFu, qp[6].x != 0.f);
          inv2[0] = make_float2(i0.x, i0.y);
          inv2[1] = make_float2(i0.z, i0.w);
          inv2[2] = make_float2(i1.x, i1.y);
          inv2[3] = make_float2(i1.z, i1.w);
          zm2[0] = make_float2(z0.x, z0.y);
          zm2[1] = make_float2(z0.z, z0.w);
          zm2[2] = make_float2(z1.x, z1.y);
          zm2[3] = make_float2(z1.z, z1.w);
          nstep2[0] = make_float2(-s0.x, -s0.y);
          nstep2[1] = make_float2(-s0.z, -s0.w);
          nstep2[2] = make_float2(-s1.x, -s1.y);
          nstep2[3] = make_float2(-s1.z, -s1.w);
#pragma unroll
          for (int j = 0; j < 4; ++j) nzm2[j] = make_float2(-zm2[j].x, -zm2[j].y);
        }
        const float* srow = reinterpret_cast<const float*>(side) + rg * 8;
        const float* rrow = reinterpret_cast<const float*>(side + kSBytes) + rg * 8;
        uint8_t* wrow = smem + kOffB + s * kBBytes + h * (kBK * 128) + (rg * 8) * 128;
        if (clampw) {
#pragma unroll
          for (int half = 0; half < 2; ++half)
            produce4<true>(wrow + half * 4 * 128, c8, half, *reinterpret_cast<const float4*>(srow + half * 4),
                           *reinterpret_cast<const float4*>(rrow + half * 4), inv2, zm2, nzm2, nstep2, lo, hi);
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half)
            produce4<false>(wrow + half * 4 * 128, c8, half, *reinterpret_cast<const float4*>(srow + half * 4),
                            *reinterpret_cast<const float4*>(rrow + half * 4), inv2, zm2, nzm2, nstep2, lo, hi);
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

// ------------------------------------------------------------------ host side
cudaError_t encode_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, CUtensorMapDataType dt,
                       int rank, const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                       const cuuint32_t* box, CUtensorMapSwizzle sw) {
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int search_fused_m_tiles(int64_t N) {
  return static_cast<int>(2 * ((N + 2 * kStack * kSubRows - 1) / (2 * kStack * kSubRows)));
}

cudaError_t launch_search_fused(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, const void* W,
                                const float* s_tab, const float* r_tab, const float* qp, int64_t N, int64_t D_in,
                                int64_t D_out, int G, int group_size, int symmetric, float* partial,
                                uint32_t* status, int max_pairs, cudaStream_t stream) {
  CUtensorMap tmX, tmW, tmS, tmR, tmQ;
  cudaError_t e;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D_in), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D_in) * 2};
    const cuuint32_t box[2] = {kBK, kSubRows};
    e = encode_map(encode, &tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D_out), static_cast<cuuint64_t>(D_in)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D_out) * 2};
    const cuuint32_t box[2] = {64, kBK};
    // 128-byte swizzle: the tile lands in the tensor cores' N-major B layout
    e = encode_map(encode, &tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D_in), static_cast<cuuint64_t>(G)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D_in) * 4};
    const cuuint32_t box[2] = {kBK, 1};
    e = encode_map(encode, &tmS, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, s_tab, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    e = encode_map(encode, &tmR, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, r_tab, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  const int T = static_cast<int>(D_in / group_size);
  {
    const cuuint64_t chunks = static_cast<cuuint64_t>(D_out / kQChunkCols);
    const cuuint64_t dims[3] = {kQChunkFloats, chunks, static_cast<cuuint64_t>(G) * T};
    const cuuint64_t strides[2] = {kQChunkFloats * 4, chunks * kQChunkFloats * 4};
    const cuuint32_t box[3] = {kQChunkFloats, kHalfN / kQChunkCols, 1};
    e = encode_map(encode, &tmQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, qp, dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  FusedArgs a;
  a.N = static_cast<int>(N);
  a.D_in = static_cast<int>(D_in);
  a.D_out = static_cast<int>(D_out);
  a.G = G;
  a.T = T;
  a.group_size = group_size;
  a.m_blocks = static_cast<int>((N + 2 * kStack * kSubRows - 1) / (2 * kStack * kSubRows));
  a.n_blocks = static_cast<int>((D_out + kPairN - 1) / kPairN);
  a.num_tiles = G * a.m_blocks * a.n_blocks;
  a.m_tiles = 2 * a.m_blocks;
  {
    // super-blocks: about 32 MB of X rows and 48 MB of W columns with their
    // parameter rows, together well inside the 126 MB L2
    const double x_band = 2.0 * kStack * kSubRows * 2.0 * static_cast<double>(D_in);
    const double w_blk = static_cast<double>(D_in) * kPairN * 2.0 +
                         static_cast<double>(G) * T * (kPairN / kQChunkCols) * kQChunkFloats * 4.0;
    a.sb_m = static_cast<int>(std::min<double>(a.m_blocks, std::max(1.0, std::floor(32e6 / x_band))));
    a.sb_n = static_cast<int>(std::min<double>(a.n_blocks, std::max(1.0, std::floor(48e6 / w_blk))));
  }
  constexpr float kMagic = 12582912.0f;
  a.clamp_lo = symmetric ? kMagic - 7.f : kMagic;
  a.clamp_hi = symmetric ? kMagic + 7.f : kMagic + 15.f;
  a.partial = partial;
  a.status = status;

  const size_t smem = static_cast<size_t>(kSmemBytes) + 1024;
  e = cudaFuncSetAttribute(search_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int pairs = max_pairs;
  if (pairs > a.num_tiles) pairs = a.num_tiles;
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, search_fused_kernel, tmX, tmW, tmS, tmR, tmQ, a);
}

// Number of CTA pairs that can be resident at once (one pair per two SMs).
cudaError_t search_fused_max_pairs(int* pairs) {
  const size_t smem = static_cast<size_t>(kSmemBytes) + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(search_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, search_fused_kernel, &cfg);
  if (e != cudaSuccess) return e;
  *pairs = n;
  return cudaSuccess;
}

}  // namespace awqdev
