// Plain tensor-core GEMM (sm_103a, tcgen05 + TMA): the self-test of the
// UMMA machinery the fused search relies on (shared-memory descriptors with
// 128-byte swizzle for a K-major A and an N-major or K-major B, the
// instruction descriptor, TMEM allocation and tcgen05.ld).  One CTA computes
// a 128 x 256 tile of C = A * B:
//
//   warp 0      TMA producer: A tile (128 rows x 64 K, K-major, 128B swizzle)
//               and B tile (64 K x 256 N) per stage
//   warp 1      TMEM allocation and the single-thread tcgen05.mma issue loop
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator, stored to C
//
// A 4-stage mbarrier ring connects TMA and MMA; every wait is bounded.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {

constexpr int BM = kGemmBM;
constexpr int BN = kGemmBN;
constexpr int BK = kGemmBK;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;         // 16 KB
constexpr int kBBoxBytes = 64 * BK * 2;      // 8 KB: 64 N x 64 K (N-major) or 64 N rows x 64 K (K-major)
constexpr int kBBytes = BN * BK * 2;         // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTmemCols = BN;                // fp32 accumulator 128 lanes x 256 columns
constexpr int kGemmThreads = 192;

static size_t gemm_smem_bytes() { return static_cast<size_t>(kStages) * kStageBytes + 1024; }

struct GemmArgs {
  int M, N, K;
  float* out;
  uint32_t* status;
};

template <int B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM;
  const int num_kb = p.K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&acc_bar, 1);
    abort_sh = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort_flag = &abort_sh;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int issued = 0;
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = (kb / kStages) & 1;
      if (kb >= kStages && !mbar_wait(&empty_bar[s], ph ^ 1, p.status, abort_flag)) break;
      mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
      tma_load_2d(sA + s * kABytes, &tmA, &full_bar[s], kb * BK, m0);
      if (B_MN) {
#pragma unroll
        for (int i = 0; i < BN / 64; ++i)
          tma_load_2d(sB + s * kBBytes + i * kBBoxBytes, &tmB, &full_bar[s], n0 + 64 * i, kb * BK);
      } else {
        tma_load_2d(sB + s * kBBytes, &tmB, &full_bar[s], kb * BK, n0);
      }
      ++issued;
    }
    if (*abort_flag) {
      // drain: wait (bounded) for the loads still in flight into this CTA
      for (int kb = issued - kStages; kb < issued; ++kb) {
        if (kb < 0) continue;
        mbar_wait(&full_bar[kb % kStages], (kb / kStages) & 1, nullptr, nullptr);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, B_MN);
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = (kb / kStages) & 1;
      if (!mbar_wait(&full_bar[s], ph, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t a_addr = smem_u32(sA + s * kABytes);
      const uint32_t b_addr = smem_u32(sB + s * kBBytes);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        // A: K-major SW128, 8-row atoms 1024 B apart; K step of 16 = +32 B
        const uint64_t ad = sdesc_sw128(a_addr + kk * 32, 16, 1024);
        // B N-major SW128: 64-wide N chunks kBBoxBytes apart (LBO), 8-row K
        //   groups 1024 B apart (SBO); K step of 16 = two K groups = +2048 B.
        // B K-major SW128: like A, 256 N rows.
        const uint64_t bd = B_MN ? sdesc_sw128(b_addr + kk * 2048, kBBoxBytes, 1024)
                                 : sdesc_sw128(b_addr + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      umma_commit(&empty_bar[s]);
    }
    umma_commit(&acc_bar);
  } else if (warp >= 2) {
    // ---------------- epilogue (TMEM lane quarter = warp % 4)
    const int q = warp & 3;
    const bool ok = mbar_wait(&acc_bar, 0, p.status, abort_flag);
    tc_fence_after();
    if (ok) {
      const int row = m0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c), v);
        if (row < p.M) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (n0 + c + i < p.N) p.out[static_cast<int64_t>(row) * p.N + n0 + c + i] = v[i];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
static cudaError_t encode_2d_bf16(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base,
                                  uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int B_MN>
static cudaError_t launch_gemm_impl(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* A, const void* B,
                                    int64_t M, int64_t N, int64_t K, float* out, uint32_t* status, cudaStream_t stream) {
  CUtensorMap tmA, tmB;
  cudaError_t e = encode_2d_bf16(encode, &tmA, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), BK, BM);
  if (e != cudaSuccess) return e;
  if (B_MN)
    e = encode_2d_bf16(encode, &tmB, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), 64, BK);
  else
    e = encode_2d_bf16(encode, &tmB, B, static_cast<uint64_t>(K), static_cast<uint64_t>(N), BK, BN);
  if (e != cudaSuccess) return e;
  const size_t smem = gemm_smem_bytes();
  e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  GemmArgs a;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.out = out;
  a.status = status;
  const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + BM - 1) / BM), 1);
  gemm_bf16_tc_kernel<B_MN><<<grid, kGemmThreads, smem, stream>>>(tmA, tmB, a);
  return cudaGetLastError();
}

cudaError_t launch_gemm_store(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* A, const void* B, int b_mn_major,
                              int64_t M, int64_t N, int64_t K, float* C, uint32_t* status, cudaStream_t stream) {
  if (b_mn_major) return launch_gemm_impl<1>(encode, A, B, M, N, K, C, status, stream);
  return launch_gemm_impl<0>(encode, A, B, M, N, K, C, status, stream);
}

}  // namespace awqdev
