// Self-test of the abort path of the CTA-pair kernels: what happens when a
// bounded mbarrier wait expires.
//
// The product kernels (search, W4A16 product) run as tcgen05 CTA pairs whose
// roles wait on one another through mbarriers.  Every wait is bounded; when
// one expires the kernel records AWQ_ERR_TIMEOUT in the status word and
// raises a CTA-local abort flag that every role polls, roles leave their
// loops, a named barrier with a reduction lets a group of warps agree on
// leaving, loaders wait (bounded) for the bulk copies they still have in
// flight, both CTAs of the pair meet at one cluster barrier, and the warp
// that allocated TMEM frees it.  This kernel runs that protocol with the same
// helpers on barriers that never receive an arrival, with a short wait limit,
// so that a test can drive a wait to expiry and then check that the status
// word says so, that TMEM was freed and that the device is still usable.
//
// Roles of each CTA (256 threads), as in the search:
//   warp 0      loader: one 4 KB bulk copy into shared memory, then a wait
//               for a free stage that never comes; drains its copy on leaving
//   warp 1      TMEM allocation for the pair (32 columns); waits for an
//               accumulator that is never committed
//   warps 2-3   epilogue: wait for the accumulator, agree on leaving through
//               a named barrier with an OR reduction
//   warps 4-7   producers: wait for an input stage that never lands
// The peer CTA cannot see this CTA's abort flag: it times out on its own.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace awqdev {
namespace {

constexpr int kAbortThreads = 256;
constexpr int kAbortCopyBytes = 4096;
constexpr uint32_t kAbortTmemCols = 32;

// record[0]: CTAs that reached the end and freed TMEM; record[1]: CTAs in
// which a wait expired (the abort flag is raised only then); record[2]: the
// largest time (us) a CTA spent from its start to its end; record[3]: CTAs
// whose bulk copy landed intact.
__global__ void __launch_bounds__(kAbortThreads, 1)
    abort_selftest_kernel(const uint8_t* __restrict__ src, uint64_t limit_ns, uint32_t* status,
                          uint32_t* record) {
  __shared__ __align__(128) uint8_t stage[kAbortCopyBytes];
  __shared__ __align__(8) uint64_t load_bar, empty_bar, acc_full_bar, wfull_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t t_start = globaltimer_ns();

  if (threadIdx.x == 0) {
    mbar_init(&load_bar, 1);
    mbar_init(&empty_bar, 1);     // never arrived on
    mbar_init(&acc_full_bar, 1);  // never committed
    mbar_init(&wfull_bar, 1);     // never lands
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, kAbortTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  volatile int* abort_flag = &abort_sh;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&load_bar, kAbortCopyBytes);
      bulk_copy_g2s(stage, src, kAbortCopyBytes, &load_bar);
      // the next stage is never freed: leave on the abort flag or on expiry
      mbar_wait(&empty_bar, 0, status, abort_flag, limit_ns);
      // the copy in flight lands before the CTA moves on (default bound)
      mbar_wait(&load_bar, 0, nullptr, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) mbar_wait(&acc_full_bar, 0, status, abort_flag, limit_ns);
  } else if (warp < 4) {
    // epilogue warps: one wait each, then agree on leaving
    for (int it = 0; it < 4; ++it) {
      const bool ok = mbar_wait(&acc_full_bar, 0, status, abort_flag, limit_ns);
      if (named_bar_or(1, 64, !ok || *abort_flag)) break;
    }
  } else {
    for (int it = 0; it < 4 && !*abort_flag; ++it)
      if (!mbar_wait(&wfull_bar, 0, status, abort_flag, limit_ns)) break;
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no arrival of one CTA may target an exited peer
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kAbortTmemCols);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // the abort flag is raised only by a wait of this CTA that expired
    if (*abort_flag) atomicAdd(&record[1], 1u);
    bool intact = true;
    for (int i = 0; i < kAbortCopyBytes; ++i) intact &= stage[i] == src[i];
    if (intact) atomicAdd(&record[3], 1u);
    atomicMax(&record[2], static_cast<uint32_t>((globaltimer_ns() - t_start) / 1000u));
    atomicAdd(&record[0], 1u);
  }
}

}  // namespace

cudaError_t launch_abort_selftest(const void* src, uint64_t limit_ns, int pairs, uint32_t* status, uint32_t* record,
                                  cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(kAbortThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, abort_selftest_kernel, static_cast<const uint8_t*>(src), limit_ns, status, record);
}

}  // namespace awqdev
