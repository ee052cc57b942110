// awq_act_stats_noalloc: the activation statistic for callers that cannot
// allocate device memory.  The per-slice partial sums, the per-chunk tickets
// and the status word that awq_act_stats keeps in the caller's workspace live
// here in one file-scope device array instead, so the caller passes only X
// and the output vector.
#include <mutex>

#include "../../include/awq.h"
#include "internal.h"

namespace {

// Layout of the array: a 256-byte header (status word at word 0) | one ticket
// counter per 256-channel chunk | 4 MiB of fp32 row-slice partial sums.  Every
// device that loads the library holds it until the process exits.  The row-
// slice plan of the statistic uses at most max(1, 296 / chunks) slices, so
// splits * D_in <= max(D_in, 296 * 256) floats: every D_in up to
// kNoAllocScratchFloats fits.
constexpr int64_t kNoAllocScratchFloats = int64_t(1) << 20;
constexpr int64_t kNoAllocHeaderWords = 64;
constexpr int64_t kNoAllocTicketWords = kNoAllocScratchFloats / 256;  // one per 256-channel chunk
static __device__ __align__(256) float g_stats_scratch[kNoAllocHeaderWords + kNoAllocTicketWords +
                                                       kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct DeviceScratch {
  unsigned long long ctx_id;  // the CUDA context the address belongs to
  float* ptr;                 // device address of g_stats_scratch in it
};
DeviceScratch g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// ID of the context current on this thread (0 when none is current yet).
awq_status current_context_id(unsigned long long* id) {
  if (!g_ctx_get_current || !g_ctx_get_id) {
    void* p = nullptr;
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r1, r2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) != cudaSuccess ||
        r1 != cudaDriverEntryPointSuccess || !p ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) != cudaSuccess ||
        r2 != cudaDriverEntryPointSuccess || !q)
      return AWQ_ERR_CUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(q);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return AWQ_ERR_CUDA;
  *id = 0;
  if (ctx && g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return AWQ_ERR_CUDA;
  return AWQ_OK;
}

// Once per device and context, with that device current: resolve the array's
// device address.  A context that was destroyed and created again (for
// example after cudaDeviceReset) has a new ID, so the address is resolved
// again in it.
awq_status scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AWQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return AWQ_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  unsigned long long id = 0;
  awq_status st = current_context_id(&id);
  if (st != AWQ_OK) return st;
  DeviceScratch& d = g_scratch[dev];
  if (!d.ptr || id == 0 || id != d.ctx_id) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return AWQ_ERR_CUDA;
    if (major != 10 || minor != 3) return AWQ_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stats_scratch) != cudaSuccess || p == nullptr) return AWQ_ERR_CUDA;
    // the lookup makes the device's primary context current if none was
    st = current_context_id(&id);
    if (st != AWQ_OK) return st;
    d.ptr = static_cast<float*>(p);
    d.ctx_id = id;
  }
  *out = d.ptr;
  return AWQ_OK;
}

}  // namespace

extern "C" awq_status awq_act_stats_noalloc(const void* X, int64_t N, int64_t D_in, int64_t ldx, float* mean_abs,
                                            awq_stream_t stream) {
  if (N < 1 || D_in < 0) return AWQ_ERR_SHAPE;
  if (D_in == 0) return AWQ_OK;
  if (D_in > kNoAllocScratchFloats) return AWQ_ERR_SHAPE;
  if (!X || !mean_abs) return AWQ_ERR_INVALID_ARG;
  if (ldx < D_in || D_in % 8 != 0 || ldx % 8 != 0 || N > INT32_MAX) return AWQ_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(X) % 16) != 0 || (reinterpret_cast<uintptr_t>(mean_abs) % 4) != 0)
    return AWQ_ERR_ALIGNMENT;
  // Same row-slice plan as awq_act_stats, so both entry points sum in the same
  // order and give the same bits.
  int splits = 1;
  int64_t rps = 0;
  awqdev::stats_plan(N, D_in, &splits, &rps);
  if (static_cast<int64_t>(splits) * D_in > kNoAllocScratchFloats) return AWQ_ERR_SHAPE;  // see the bound above
  float* scratch = nullptr;
  awq_status st = scratch_for_current_device(&scratch);
  if (st != AWQ_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  st = awqdev::tensor_map_encoder(&encode);
  if (st != AWQ_OK) return st;

  // The status word and the ticket counters must start at zero (the kernel
  // leaves the tickets zero, but clearing them here keeps each call
  // self-contained); every partial the final sums read is rewritten by this
  // call.  A wait that gives up sets the status word, and the means of its
  // chunk are then written as NaN; a non-finite X shows up as a non-finite
  // mean on its own.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = reinterpret_cast<uint32_t*>(scratch);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(scratch + kNoAllocHeaderWords);
  const int64_t chunks = awqdev::stats_chunks(D_in);
  if (cudaMemsetAsync(scratch, 0, static_cast<size_t>(kNoAllocHeaderWords + chunks) * sizeof(float), s) !=
      cudaSuccess)
    return AWQ_ERR_CUDA;
  const cudaError_t e = awqdev::launch_act_stats(
      encode, X, N, D_in, ldx, mean_abs, nullptr, nullptr, scratch + kNoAllocHeaderWords + kNoAllocTicketWords,
      nullptr, tickets, splits, rps, status, 1, s);
  return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA;
}
