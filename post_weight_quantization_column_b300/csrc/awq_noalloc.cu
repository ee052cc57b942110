// awq_act_stats_noalloc: the activation statistic for callers that cannot
// allocate device memory.  The per-slice partial sums that awq_act_stats
// keeps in the caller's workspace live here in one file-scope device array
// instead, so the caller passes only X and the output vector.
#include <mutex>

#include "../../include/awq.h"
#include "internal.h"

namespace {

// 4 MiB of fp32 partial sums plus 16 KiB of per-chunk ticket counters in
// front of them, held by every device that loads the library until the
// process exits.  One slice of D_in channels must fit, so D_in is limited to
// kNoAllocScratchFloats.
constexpr int64_t kNoAllocScratchFloats = int64_t(1) << 20;
constexpr int64_t kNoAllocTicketWords = kNoAllocScratchFloats / 256;  // one per 256-channel chunk
static __device__ __align__(256) float g_stats_scratch[kNoAllocTicketWords + kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_scratch_ptr[kMaxDevices];  // device address of g_stats_scratch, per device

// Once per device, with that device current: resolve the array's device address.
awq_status scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AWQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return AWQ_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_scratch_ptr[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return AWQ_ERR_CUDA;
    if (major != 10 || minor != 3) return AWQ_ERR_UNSUPPORTED_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stats_scratch) != cudaSuccess || p == nullptr) return AWQ_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
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
  float* scratch = nullptr;
  awq_status st = scratch_for_current_device(&scratch);
  if (st != AWQ_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  st = awqdev::tensor_map_encoder(&encode);
  if (st != AWQ_OK) return st;

  // Same row-slice plan as awq_act_stats, so both entry points sum in the same
  // order (that plan keeps splits * D_in below the array for every allowed
  // D_in); should it ever not fit, use fewer, longer slices.
  int splits = 1;
  int64_t rps = 0;
  awqdev::stats_plan(N, D_in, &splits, &rps);
  if (static_cast<int64_t>(splits) * D_in > kNoAllocScratchFloats) {
    const int64_t max_splits = kNoAllocScratchFloats / D_in;
    rps = (N + max_splits - 1) / max_splits;
    rps = (rps + awqdev::kStatsBoxRows - 1) / awqdev::kStatsBoxRows * awqdev::kStatsBoxRows;
    splits = static_cast<int>((N + rps - 1) / rps);
  }
  // Every partial the final sums read is rewritten by this call; the ticket
  // counters must start at zero (the kernel leaves them zero, and the array
  // starts zeroed, but clearing them here keeps each call self-contained).
  // There is no status word: a non-finite X shows up as a non-finite mean.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(scratch);
  const int64_t chunks = awqdev::stats_chunks(D_in);
  if (cudaMemsetAsync(tickets, 0, static_cast<size_t>(chunks) * sizeof(unsigned int), s) != cudaSuccess)
    return AWQ_ERR_CUDA;
  const cudaError_t e = awqdev::launch_act_stats(encode, X, N, D_in, ldx, mean_abs, nullptr, nullptr,
                                                 scratch + kNoAllocTicketWords, nullptr, tickets, splits, rps,
                                                 nullptr, s);
  return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA;
}
