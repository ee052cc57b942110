// C ABI of the AWQ calibration hot path: argument validation, workspace
// layout and kernel launch order.  Every function validates on the host
// first and makes no CUDA call when validation fails.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/awq.h"
#include "../../include/awq_profile.h"
#include "../../include/awq_selftest.h"
#include "internal.h"

using namespace awqdev;

namespace {

constexpr size_t kHeaderBytes = 256;  // status word at offset 0, reduction ticket at offset 4
constexpr int kMaxDevices = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- device / driver state
std::mutex g_mu;
int g_arch_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other
int g_pairs[kMaxDevices];    // resident CTA pairs of the fused search (0 = not queried)
int g_w4a16_pairs[kMaxDevices];  // resident CTA pairs of the W4A16 product (0 = not queried)
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

awq_status check_device(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return AWQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return AWQ_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return AWQ_ERR_CUDA;
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_arch_ok[dev] != 1) return AWQ_ERR_UNSUPPORTED_DEVICE;
  if (dev_out) *dev_out = dev;
  return AWQ_OK;
}

awq_status get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
      return AWQ_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = g_encode;
  return AWQ_OK;
}

awq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA; }

awq_status get_w4a16_pairs(int dev, int* pairs) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_w4a16_pairs[dev] == 0) {
    int n = 0;
    if (w4a16_max_pairs(&n) != cudaSuccess || n < 1) return AWQ_ERR_CUDA;
    g_w4a16_pairs[dev] = n;
  }
  *pairs = g_w4a16_pairs[dev];
  return AWQ_OK;
}

awq_status get_pairs(int dev, int* pairs) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_pairs[dev] == 0) {
    int n = 0;
    if (search_fused_max_pairs(&n) != cudaSuccess || n < 1) return AWQ_ERR_CUDA;
    g_pairs[dev] = n;
  }
  *pairs = g_pairs[dev];
  return AWQ_OK;
}

// ---------------------------------------------------------------- optional event timing
struct ProfRecord {
  std::string name;
  cudaEvent_t start, stop;
};
struct Profiler {
  std::mutex mu;
  bool enabled = false;
  std::vector<cudaEvent_t> pool;
  std::vector<ProfRecord> records;
  cudaEvent_t take() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
};
Profiler g_prof;

// Brackets one launcher call with events on its stream while timing is on.
class ProfScope {
 public:
  ProfScope(const char* name, cudaStream_t s) : name_(name), s_(s) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (!g_prof.enabled) return;
    start_ = g_prof.take();
    stop_ = g_prof.take();
    if (start_ && stop_ && cudaEventRecord(start_, s_) == cudaSuccess) active_ = true;
  }
  ~ProfScope() {
    if (!active_) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (cudaEventRecord(stop_, s_) == cudaSuccess) g_prof.records.push_back({name_, start_, stop_});
  }

 private:
  const char* name_;
  cudaStream_t s_;
  cudaEvent_t start_ = nullptr, stop_ = nullptr;
  bool active_ = false;
};

awq_status validate_cfg(const awq_cfg* cfg) {
  if (!cfg) return AWQ_ERR_INVALID_ARG;
  if (cfg->bits != 4) return AWQ_ERR_INVALID_ARG;
  if (cfg->group_size != 64 && cfg->group_size != 128 && cfg->group_size != 256) return AWQ_ERR_INVALID_ARG;
  if (cfg->symmetric != 0 && cfg->symmetric != 1) return AWQ_ERR_INVALID_ARG;
  if (!std::isfinite(cfg->act_floor) || cfg->act_floor < 0.f) return AWQ_ERR_INVALID_ARG;
  return AWQ_OK;
}

uint32_t* status_word(void* ws) { return static_cast<uint32_t*>(ws); }

// ---------------------------------------------------------------- layouts
// act_stats workspace: header (status word) | tickets [stats_chunks] |
// partial sums [splits][D_in] | partial maxima [splits][D_in]
size_t stats_ticket_bytes(int64_t D_in) { return align_up(static_cast<size_t>(stats_chunks(D_in)) * 4, 256); }
size_t stats_partial_bytes(int64_t N, int64_t D_in) {
  int splits = 1;
  int64_t rps = 0;
  stats_plan(N, D_in, &splits, &rps);
  return align_up(static_cast<size_t>(splits) * static_cast<size_t>(D_in) * 4, 256);
}
size_t stats_ws_bytes(int64_t N, int64_t D_in) {
  return kHeaderBytes + stats_ticket_bytes(D_in) + 2 * stats_partial_bytes(N, D_in);
}

struct SearchLayout {
  size_t s_tab, r_tab, qp, partial, col, blk, total;
  int m_tiles;
};

SearchLayout search_layout(int64_t N, int64_t D_in, int64_t D_out, int G, int group_size) {
  SearchLayout L;
  const size_t g = static_cast<size_t>(G);
  const size_t din = static_cast<size_t>(D_in), dout = static_cast<size_t>(D_out);
  L.m_tiles = search_fused_m_tiles(N);
  size_t off = kHeaderBytes;
  L.s_tab = off;
  off = align_up(off + g * din * 4, 256);
  L.r_tab = off;
  off = align_up(off + g * din * 4, 256);
  L.qp = off;
  off = align_up(off + qparam_floats(G, D_in / group_size, D_out) * 4, 256);
  L.partial = off;
  off = align_up(off + g * static_cast<size_t>(L.m_tiles) * dout * 4, 256);
  L.col = off;
  off = align_up(off + g * dout * 8, 256);
  L.blk = off;
  off = align_up(off + g * static_cast<size_t>(reduce_blocks(D_out)) * 8, 256);
  L.total = off;
  return L;
}

// Offset of the group-parameter table inside a search workspace (the layout
// before it depends only on D_in and G).
size_t search_qp_offset(int64_t D_in, int G) {
  const size_t g = static_cast<size_t>(G), din = static_cast<size_t>(D_in);
  size_t off = align_up(kHeaderBytes + g * din * 4, 256);
  return align_up(off + g * din * 4, 256);
}

awq_status validate_search_shape(int64_t N, int64_t D_in, int64_t D_out, int32_t G, const awq_cfg* cfg) {
  awq_status st = validate_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (G < 1 || G > kMaxGrid) return AWQ_ERR_SHAPE;
  if (N < 1 || D_in < 1 || D_out < 1) return AWQ_ERR_SHAPE;
  if (D_in % cfg->group_size != 0 || D_out % 8 != 0) return AWQ_ERR_SHAPE;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (N > lim || D_in > lim / G || D_out > lim) return AWQ_ERR_SHAPE;
  return AWQ_OK;
}

}  // namespace

namespace awqdev {
awq_status tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) { return get_encode(fn); }
}  // namespace awqdev

extern "C" {

const char* awq_status_string(awq_status s) {
  switch (s) {
    case AWQ_OK: return "AWQ_OK";
    case AWQ_ERR_INVALID_ARG: return "AWQ_ERR_INVALID_ARG: null pointer or invalid configuration value";
    case AWQ_ERR_SHAPE: return "AWQ_ERR_SHAPE: sizes out of range or not divisible as required";
    case AWQ_ERR_ALIGNMENT: return "AWQ_ERR_ALIGNMENT: pointer or leading dimension misaligned";
    case AWQ_ERR_WORKSPACE: return "AWQ_ERR_WORKSPACE: workspace too small";
    case AWQ_ERR_UNSUPPORTED_DEVICE: return "AWQ_ERR_UNSUPPORTED_DEVICE: current device is not sm_103";
    case AWQ_ERR_CUDA: return "AWQ_ERR_CUDA: a CUDA call failed";
    case AWQ_ERR_RANGE: return "AWQ_ERR_RANGE: quantisation step does not fit in fp16";
    case AWQ_ERR_NONFINITE: return "AWQ_ERR_NONFINITE: NaN or infinity in an input";
    case AWQ_ERR_TIMEOUT: return "AWQ_ERR_TIMEOUT: a bounded device wait expired";
  }
  return "AWQ_ERR_UNKNOWN";
}

awq_status awq_workspace_status(const void* ws, awq_stream_t stream) {
  if (!ws) return AWQ_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  e = cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  return static_cast<awq_status>(word);
}

// ------------------------------------------------------------------ stats
awq_status awq_act_stats_workspace_size(int64_t N, int64_t D_in, size_t* bytes) {
  if (!bytes) return AWQ_ERR_INVALID_ARG;
  if (N < 1 || D_in < 0) return AWQ_ERR_SHAPE;
  *bytes = stats_ws_bytes(N, D_in);
  return AWQ_OK;
}

namespace {
// One pass of the statistic kernel over X: the mean into mean_abs, or (when
// sum_abs is given) the float64 column sums added to sum_abs; max_abs, when
// given, takes the running maximum of |x|.
awq_status run_act_stats(const void* X, int64_t N, int64_t D_in, int64_t ldx, float* mean_abs, double* sum_abs,
                         float* max_abs, void* ws, size_t ws_bytes, awq_stream_t stream, const char* name) {
  if (N < 1 || D_in < 0) return AWQ_ERR_SHAPE;
  if (D_in == 0) return AWQ_OK;
  if (!X || (!mean_abs && !sum_abs) || !ws) return AWQ_ERR_INVALID_ARG;
  if (ldx < D_in || D_in % 8 != 0 || ldx % 8 != 0 || N > INT32_MAX || D_in > INT32_MAX) return AWQ_ERR_SHAPE;
  if (!aligned(X, 16) || (mean_abs && !aligned(mean_abs, 4)) || (sum_abs && !aligned(sum_abs, 8)) ||
      (max_abs && !aligned(max_abs, 4)) || !aligned(ws, 256))
    return AWQ_ERR_ALIGNMENT;
  if (ws_bytes < stats_ws_bytes(N, D_in)) return AWQ_ERR_WORKSPACE;
  awq_status st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  st = get_encode(&encode);
  if (st != AWQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int splits = 1;
  int64_t rps = 0;
  stats_plan(N, D_in, &splits, &rps);
  // status word and the ticket counters start at zero
  const size_t tb = stats_ticket_bytes(D_in);
  if (cudaMemsetAsync(ws, 0, kHeaderBytes + tb, s) != cudaSuccess) return AWQ_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(ws);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(base + kHeaderBytes);
  float* partial = reinterpret_cast<float*>(base + kHeaderBytes + tb);
  float* partial_max = reinterpret_cast<float*>(base + kHeaderBytes + tb + stats_partial_bytes(N, D_in));
  ProfScope prof(name, s);
  return from_cuda(launch_act_stats(encode, X, N, D_in, ldx, mean_abs, sum_abs, max_abs, partial, partial_max,
                                    tickets, splits, rps, status_word(ws), 0, s));
}
}  // namespace

awq_status awq_act_stats(const void* X, int64_t N, int64_t D_in, int64_t ldx, float* mean_abs, void* ws,
                         size_t ws_bytes, awq_stream_t stream) {
  if (N >= 1 && D_in > 0 && !mean_abs) return AWQ_ERR_INVALID_ARG;
  return run_act_stats(X, N, D_in, ldx, mean_abs, nullptr, nullptr, ws, ws_bytes, stream, "act_stats");
}

awq_status awq_act_stats_accumulate(const void* X, int64_t N, int64_t D_in, int64_t ldx, double* sum_abs,
                                    float* max_abs, void* ws, size_t ws_bytes, awq_stream_t stream) {
  if (N >= 1 && D_in > 0 && !sum_abs) return AWQ_ERR_INVALID_ARG;
  return run_act_stats(X, N, D_in, ldx, nullptr, sum_abs, max_abs, ws, ws_bytes, stream, "act_stats_accumulate");
}

awq_status awq_act_stats_finalize(const double* sum_abs, int64_t rows, int64_t D_in, float* mean_abs,
                                  awq_stream_t stream) {
  if (rows < 1 || D_in < 0) return AWQ_ERR_SHAPE;
  if (D_in == 0) return AWQ_OK;
  if (!sum_abs || !mean_abs) return AWQ_ERR_INVALID_ARG;
  if (!aligned(sum_abs, 8) || !aligned(mean_abs, 4)) return AWQ_ERR_ALIGNMENT;
  awq_status st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  return from_cuda(launch_stats_finalize(sum_abs, rows, D_in, mean_abs, reinterpret_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ search
awq_status awq_search_workspace_size(int64_t N, int64_t D_in, int64_t D_out, int32_t G, const awq_cfg* cfg,
                                     size_t* bytes) {
  if (!bytes) return AWQ_ERR_INVALID_ARG;
  awq_status st = validate_search_shape(N, D_in, D_out, G, cfg);
  if (st != AWQ_OK) return st;
  *bytes = search_layout(N, D_in, D_out, G, cfg->group_size).total;
  return AWQ_OK;
}

namespace {
// The search on "X" [N, D_in] (the calibration rows, or the Gram factor R
// with N = D_in rows): scale table, group parameters, fused search, reduce.
awq_status run_search(const void* X, const void* W, int64_t N, int64_t D_in, int64_t D_out, const float* mean_abs,
                      const AlphaGrid& ag, int32_t G, const awq_cfg* cfg, double* losses, int32_t* best_idx,
                      float* s_star, double* col_losses, void* ws, int dev, PFN_cuTensorMapEncodeTiled_v12000 encode,
                      cudaStream_t s) {
  const SearchLayout L = search_layout(N, D_in, D_out, G, cfg->group_size);
  int pairs = 0;
  awq_status st = get_pairs(dev, &pairs);
  if (st != AWQ_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* status = status_word(ws);
  float* s_tab = reinterpret_cast<float*>(base + L.s_tab);
  float* r_tab = reinterpret_cast<float*>(base + L.r_tab);
  float* qp = reinterpret_cast<float*>(base + L.qp);
  float* partial = reinterpret_cast<float*>(base + L.partial);
  double* col = col_losses ? col_losses : reinterpret_cast<double*>(base + L.col);
  cudaError_t e;
  {
    ProfScope prof("scale_table", s);
    e = launch_scale_table(mean_abs, D_in, ag, G, cfg->act_floor, s_tab, r_tab, status, s);
  }
  if (e == cudaSuccess) {
    ProfScope prof("group_params", s);
    e = launch_group_params(W, s_tab, D_in, D_out, G, cfg->group_size, cfg->symmetric, qp, status, s);
  }
  if (e == cudaSuccess) {
    ProfScope prof("search_fused", s);
    e = launch_search_fused(encode, X, W, s_tab, r_tab, qp, N, D_in, D_out, G, cfg->group_size, cfg->symmetric,
                            partial, status, pairs, s);
  }
  if (e == cudaSuccess) {
    ProfScope prof("reduce_argmin", s);
    e = launch_reduce_losses(partial, L.m_tiles, D_out, G, col, reinterpret_cast<double*>(base + L.blk),
                             reinterpret_cast<unsigned int*>(base + 4), losses, best_idx, s_tab, D_in, s_star, status,
                             s);
  }
  return from_cuda(e);
}

awq_status search_args(const void* X, const void* W, int64_t N, int64_t D_in, int64_t D_out, const float* mean_abs,
                       const double* grid, int32_t G, const awq_cfg* cfg, double* losses, int32_t* best_idx,
                       float* s_star, double* col_losses, void* ws, AlphaGrid* ag) {
  if (!X || !W || !mean_abs || !grid || !cfg || !losses || !best_idx || !s_star || !ws) return AWQ_ERR_INVALID_ARG;
  awq_status st = validate_search_shape(N, D_in, D_out, G, cfg);
  if (st != AWQ_OK) return st;
  std::memset(ag, 0, sizeof(*ag));
  for (int k = 0; k < G; ++k) {
    if (!std::isfinite(grid[k]) || grid[k] < 0.0 || grid[k] > 1.0) return AWQ_ERR_INVALID_ARG;
    ag->a[k] = grid[k];
  }
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(ws, 256) || !aligned(mean_abs, 4) || !aligned(s_star, 4) ||
      !aligned(losses, 8) || !aligned(best_idx, 4) || (col_losses && !aligned(col_losses, 8)))
    return AWQ_ERR_ALIGNMENT;
  return AWQ_OK;
}

// Gram-form workspace: the search workspace for N = D_in rows (first, so that
// the searched pack finds its group parameters at the usual offset) | H fp32
// [D_in, D_in] | the inverse of one 64 x 64 Cholesky block (16 KB) | X^T bf16
// [D_in, ldt], later R bf16 [D_in, D_in] in the same place
struct GramLayout {
  size_t h, linv, t, total;
  int64_t ldt;
};
GramLayout gram_layout(int64_t N, int64_t D_in, int64_t D_out, int G, int group_size) {
  GramLayout L;
  L.ldt = (N + kGemmBK - 1) / kGemmBK * kGemmBK;
  L.h = align_up(search_layout(D_in, D_in, D_out, G, group_size).total, 256);
  L.linv = L.h + align_up(static_cast<size_t>(D_in) * static_cast<size_t>(D_in) * 4, 256);
  L.t = L.linv + 64 * 64 * 4;
  const size_t tb = static_cast<size_t>(D_in) * static_cast<size_t>(L.ldt > D_in ? L.ldt : D_in) * 2;
  L.total = L.t + align_up(tb, 256);
  return L;
}
}  // namespace

awq_status awq_search(const void* X, const void* W, int64_t N, int64_t D_in, int64_t D_out, const float* mean_abs,
                      const double* grid, int32_t G, const awq_cfg* cfg, double* losses, int32_t* best_idx,
                      float* s_star, double* col_losses, void* ws, size_t ws_bytes, awq_stream_t stream) {
  AlphaGrid ag;
  awq_status st = search_args(X, W, N, D_in, D_out, mean_abs, grid, G, cfg, losses, best_idx, s_star, col_losses, ws,
                              &ag);
  if (st != AWQ_OK) return st;
  if (ws_bytes < search_layout(N, D_in, D_out, G, cfg->group_size).total) return AWQ_ERR_WORKSPACE;
  int dev = 0;
  st = check_device(&dev);
  if (st != AWQ_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  st = get_encode(&encode);
  if (st != AWQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // status word and the reduction's ticket counter
  if (cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), s) != cudaSuccess) return AWQ_ERR_CUDA;
  return run_search(X, W, N, D_in, D_out, mean_abs, ag, G, cfg, losses, best_idx, s_star, col_losses, ws, dev,
                    encode, s);
}

awq_status awq_search_block_losses(const void* ws, size_t ws_bytes, int64_t N, int64_t D_in, int64_t D_out,
                                  int32_t G, const awq_cfg* cfg, double* blk, awq_stream_t stream) {
  awq_status st = validate_search_shape(N, D_in, D_out, G, cfg);
  if (st != AWQ_OK) return st;
  if (!ws || !blk) return AWQ_ERR_INVALID_ARG;
  if (!aligned(ws, 256) || !aligned(blk, 8)) return AWQ_ERR_ALIGNMENT;
  const SearchLayout L = search_layout(N, D_in, D_out, G, cfg->group_size);
  if (ws_bytes < L.total) return AWQ_ERR_WORKSPACE;
  st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  const size_t bytes = static_cast<size_t>(G) * static_cast<size_t>(reduce_blocks(D_out)) * sizeof(double);
  return from_cuda(cudaMemcpyAsync(blk, static_cast<const uint8_t*>(ws) + L.blk, bytes, cudaMemcpyDeviceToDevice,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

awq_status awq_search_select(const double* blk, int64_t nb, int32_t G, void* ws, size_t ws_bytes, int64_t N,
                             int64_t D_in, int64_t D_out, const awq_cfg* cfg, double* losses, int32_t* best_idx,
                             float* s_star, awq_stream_t stream) {
  awq_status st = validate_search_shape(N, D_in, D_out, G, cfg);
  if (st != AWQ_OK) return st;
  if (nb < 1 || nb > (int64_t(1) << 40)) return AWQ_ERR_SHAPE;
  if (!blk || !ws || !losses || !best_idx || !s_star) return AWQ_ERR_INVALID_ARG;
  if (!aligned(blk, 8) || !aligned(ws, 256) || !aligned(losses, 8) || !aligned(best_idx, 4) || !aligned(s_star, 4))
    return AWQ_ERR_ALIGNMENT;
  const SearchLayout L = search_layout(N, D_in, D_out, G, cfg->group_size);
  if (ws_bytes < L.total) return AWQ_ERR_WORKSPACE;
  st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const float* s_tab = reinterpret_cast<const float*>(static_cast<const uint8_t*>(ws) + L.s_tab);
  ProfScope prof("select", cs);
  return from_cuda(launch_select_losses(blk, nb, G, losses, best_idx, s_tab, D_in, s_star, status_word(ws), cs));
}

awq_status awq_search_gram_workspace_size(int64_t N, int64_t D_in, int64_t D_out, int32_t G, const awq_cfg* cfg,
                                          size_t* bytes) {
  if (!bytes) return AWQ_ERR_INVALID_ARG;
  awq_status st = validate_search_shape(N, D_in, D_out, G, cfg);
  if (st != AWQ_OK) return st;
  if (N < D_in || D_in % 64 != 0) return AWQ_ERR_SHAPE;
  *bytes = gram_layout(N, D_in, D_out, G, cfg->group_size).total;
  return AWQ_OK;
}

awq_status awq_search_gram(const void* X, const void* W, int64_t N, int64_t D_in, int64_t D_out,
                           const float* mean_abs, const double* grid, int32_t G, const awq_cfg* cfg, double* losses,
                           int32_t* best_idx, float* s_star, double* col_losses, void* ws, size_t ws_bytes,
                           awq_stream_t stream) {
  AlphaGrid ag;
  awq_status st = search_args(X, W, N, D_in, D_out, mean_abs, grid, G, cfg, losses, best_idx, s_star, col_losses, ws,
                              &ag);
  if (st != AWQ_OK) return st;
  if (N < D_in || D_in % 64 != 0) return AWQ_ERR_SHAPE;
  if (D_in > 65535 * static_cast<int64_t>(kGemmBM)) return AWQ_ERR_SHAPE;
  const GramLayout G2 = gram_layout(N, D_in, D_out, G, cfg->group_size);
  if (ws_bytes < G2.total) return AWQ_ERR_WORKSPACE;
  int dev = 0;
  st = check_device(&dev);
  if (st != AWQ_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  st = get_encode(&encode);
  if (st != AWQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* H = reinterpret_cast<float*>(base + G2.h);
  void* T = base + G2.t;
  if (cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), s) != cudaSuccess) return AWQ_ERR_CUDA;
  cudaError_t e;
  {
    // H = X^T X from the zero-padded transpose (both operands K-major)
    ProfScope prof("gram", s);
    e = launch_transpose_x(X, N, D_in, G2.ldt, T, s);
    if (e == cudaSuccess)
      e = launch_gemm_store(encode, T, T, 0, D_in, D_in, G2.ldt, H, status_word(ws), s);
  }
  if (e == cudaSuccess) {
    ProfScope prof("cholesky", s);
    e = launch_cholesky(H, D_in, reinterpret_cast<float*>(base + G2.linv), status_word(ws), s);
    if (e == cudaSuccess) e = launch_lt_to_bf16(H, D_in, T, s);  // R = L^T over the dead transpose
  }
  if (e != cudaSuccess) return from_cuda(e);
  return run_search(T, W, D_in, D_in, D_out, mean_abs, ag, G, cfg, losses, best_idx, s_star, col_losses, ws, dev,
                    encode, s);
}

// ------------------------------------------------------------------ pack
awq_status awq_pack_workspace_size(int64_t D_in, int64_t D_out, const awq_cfg* cfg, size_t* bytes) {
  if (!bytes) return AWQ_ERR_INVALID_ARG;
  awq_status st = validate_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (D_in < 0 || D_out < 0) return AWQ_ERR_SHAPE;
  *bytes = kHeaderBytes;
  return AWQ_OK;
}

awq_status awq_quantize_pack(const void* W, const float* s, int64_t D_in, int64_t D_out, const awq_cfg* cfg,
                             uint8_t* qweight, void* scales, void* zeros, void* ws, size_t ws_bytes,
                             awq_stream_t stream) {
  awq_status st = validate_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (D_in < 0 || D_out < 0) return AWQ_ERR_SHAPE;
  if (D_in % cfg->group_size != 0 || D_out % 8 != 0) return AWQ_ERR_SHAPE;
  if (D_in / cfg->group_size > 65535) return AWQ_ERR_SHAPE;
  if (D_in == 0 || D_out == 0) return AWQ_OK;
  if (!W || !s || !qweight || !scales || !zeros || !ws) return AWQ_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(s, 4) || !aligned(qweight, 8) || !aligned(scales, 2) || !aligned(zeros, 2) ||
      !aligned(ws, 256))
    return AWQ_ERR_ALIGNMENT;
  if (ws_bytes < kHeaderBytes) return AWQ_ERR_WORKSPACE;
  int dev = 0;
  st = check_device(&dev);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), cs) != cudaSuccess) return AWQ_ERR_CUDA;
  ProfScope prof("pack", cs);
  return from_cuda(launch_pack(W, s, D_in, D_out, cfg->group_size, cfg->symmetric, qweight, scales, zeros,
                               status_word(ws), cs));
}

awq_status awq_quantize_pack_searched(const void* W, int64_t D_in, int64_t D_out, int32_t G, const awq_cfg* cfg,
                                      const void* search_ws, size_t search_ws_bytes, const int32_t* best_idx,
                                      const float* s_star, uint8_t* qweight, void* scales, void* zeros,
                                      awq_stream_t stream) {
  awq_status st = validate_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (G < 1 || G > kMaxGrid) return AWQ_ERR_SHAPE;
  if (D_in < 0 || D_out < 0) return AWQ_ERR_SHAPE;
  if (D_in % cfg->group_size != 0 || D_out % 8 != 0) return AWQ_ERR_SHAPE;
  if (D_in == 0 || D_out == 0) return AWQ_OK;
  if (!W || !search_ws || !best_idx || !s_star || !qweight || !scales || !zeros) return AWQ_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(search_ws, 256) || !aligned(best_idx, 4) || !aligned(s_star, 16) ||
      !aligned(qweight, 8) || !aligned(scales, 16) || !aligned(zeros, 16))
    return AWQ_ERR_ALIGNMENT;
  const size_t qp_off = search_qp_offset(D_in, G);
  if (search_ws_bytes < qp_off + qparam_floats(G, D_in / cfg->group_size, D_out) * 4) return AWQ_ERR_WORKSPACE;
  st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const float* qp = reinterpret_cast<const float*>(static_cast<const uint8_t*>(search_ws) + qp_off);
  ProfScope prof("pack_searched", cs);
  return from_cuda(launch_pack_searched(W, s_star, qp, best_idx, G, D_in, D_out, cfg->group_size, cfg->symmetric,
                                        qweight, scales, zeros, cs));
}

// ------------------------------------------------------------------ closed-form scale
awq_status awq_closed_form_scales(const void* W, int64_t D_in, int64_t D_out, const float* mean_abs, double alpha,
                                  const awq_cfg* cfg, float* s_out, awq_stream_t stream) {
  awq_status st = validate_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (D_in < 0 || D_out < 0 || D_out % 8 != 0) return AWQ_ERR_SHAPE;
  if (!(alpha >= 0.0 && alpha <= 1.0)) return AWQ_ERR_INVALID_ARG;
  if (D_in == 0 || D_out == 0) return AWQ_OK;
  if (!W || !mean_abs || !s_out) return AWQ_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(mean_abs, 4) || !aligned(s_out, 4)) return AWQ_ERR_ALIGNMENT;
  st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  ProfScope prof("closed_form", cs);
  return from_cuda(launch_closed_form(W, D_in, D_out, mean_abs, alpha, cfg->act_floor, s_out, cs));
}

// ------------------------------------------------------------------ the adr's greedy search
namespace {
// greedy workspace: header | current candidate index [D_in] int32 |
// partials [T][slices][kMaxGreedyCand + 1] fp32 | tickets [T]
struct GreedyLayout {
  size_t idx, partial, tickets, total;
};
GreedyLayout greedy_layout(int64_t D_in, int64_t D_out, int group_size) {
  GreedyLayout L;
  const int64_t T = D_in / group_size;
  L.idx = kHeaderBytes;
  L.partial = L.idx + align_up(static_cast<size_t>(D_in) * 4, 256);
  L.tickets = L.partial + align_up(static_cast<size_t>(T) * greedy_slices(D_out) * (kMaxGreedyCand + 1) * 4, 256);
  L.total = L.tickets + align_up(static_cast<size_t>(T) * 4, 256);
  return L;
}
awq_status validate_greedy(int64_t D_in, int64_t D_out, const awq_cfg* cfg, int32_t passes, int32_t k_min,
                           int32_t n_cand) {
  awq_status st = validate_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (D_in < 0 || D_out < 0 || D_in % cfg->group_size != 0 || D_out % 8 != 0) return AWQ_ERR_SHAPE;
  if (D_in > INT32_MAX || D_out > INT32_MAX || D_in / cfg->group_size > 65535) return AWQ_ERR_SHAPE;
  if (passes < 1 || passes > 16 || n_cand < 1 || n_cand > kMaxGreedyCand) return AWQ_ERR_INVALID_ARG;
  if (k_min > 0 || k_min + n_cand <= 0 || k_min < -60 || k_min + n_cand > 60) return AWQ_ERR_INVALID_ARG;
  return AWQ_OK;
}
}  // namespace

awq_status awq_greedy_workspace_size(int64_t D_in, int64_t D_out, const awq_cfg* cfg, size_t* bytes) {
  if (!bytes) return AWQ_ERR_INVALID_ARG;
  awq_status st = validate_greedy(D_in, D_out, cfg, 1, -10, 20);
  if (st != AWQ_OK) return st;
  *bytes = greedy_layout(D_in, D_out, cfg->group_size).total;
  return AWQ_OK;
}

awq_status awq_greedy_search(const void* W, const float* mean_abs, int64_t D_in, int64_t D_out, const awq_cfg* cfg,
                             int32_t passes, int32_t k_min, int32_t n_cand, float* s_out, int32_t* trace,
                             double* errors, void* ws, size_t ws_bytes, awq_stream_t stream) {
  awq_status st = validate_greedy(D_in, D_out, cfg, passes, k_min, n_cand);
  if (st != AWQ_OK) return st;
  if (D_in == 0 || D_out == 0) return AWQ_OK;
  if (!W || !mean_abs || !s_out || !ws) return AWQ_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(mean_abs, 4) || !aligned(s_out, 4) || (trace && !aligned(trace, 4)) ||
      (errors && !aligned(errors, 8)) || !aligned(ws, 256))
    return AWQ_ERR_ALIGNMENT;
  const GreedyLayout L = greedy_layout(D_in, D_out, cfg->group_size);
  if (ws_bytes < L.total) return AWQ_ERR_WORKSPACE;
  st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  if (cudaMemsetAsync(ws, 0, kHeaderBytes, cs) != cudaSuccess) return AWQ_ERR_CUDA;
  if (cudaMemsetAsync(base + L.tickets, 0, L.total - L.tickets, cs) != cudaSuccess) return AWQ_ERR_CUDA;
  ProfScope prof("greedy", cs);
  return from_cuda(launch_greedy(W, mean_abs, D_in, D_out, cfg->group_size, cfg->symmetric, passes, k_min, n_cand,
                                 s_out, reinterpret_cast<int*>(base + L.idx), reinterpret_cast<float*>(base + L.partial),
                                 reinterpret_cast<unsigned int*>(base + L.tickets), trace, errors, status_word(ws),
                                 cs));
}

// ------------------------------------------------------------------ W4A16 product
namespace {
// W4A16 workspace: header | (decode path) tickets [D_out/1024] | B fragments of x' [D_in/64 chunks] |
// partials [1024 + D_out/1024][M][1024]
size_t w4a16_ticket_bytes(int64_t D_out) { return align_up(static_cast<size_t>(w4a16_decode_tickets(D_out)) * 4, 256); }
size_t w4a16_xprep_bytes(int64_t D_in) { return align_up(static_cast<size_t>(w4a16_decode_xprep_bytes(D_in)), 256); }
size_t w4a16_ws_bytes(int64_t M, int64_t D_in, int64_t D_out) {
  if (M > kW4a16DecodeMaxRows) return kHeaderBytes;
  return kHeaderBytes + w4a16_ticket_bytes(D_out) + w4a16_xprep_bytes(D_in) +
         align_up(static_cast<size_t>(w4a16_decode_partial_floats(M, D_in, D_out)) * 4, 256);
}
}  // namespace

awq_status awq_w4a16_workspace_size(int64_t M, int64_t D_in, int64_t D_out, size_t* bytes) {
  if (!bytes) return AWQ_ERR_INVALID_ARG;
  if (M < 0 || D_in < 0 || D_out < 0) return AWQ_ERR_SHAPE;
  *bytes = w4a16_ws_bytes(M, D_in, D_out);
  return AWQ_OK;
}

awq_status awq_w4a16_matmul(const void* X, int64_t M, int64_t D_in, int64_t D_out, const uint8_t* qweight,
                            const void* scales, const void* zeros, const float* s, const awq_cfg* cfg, void* Y,
                            void* ws, size_t ws_bytes, awq_stream_t stream) {
  awq_status st = validate_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (M < 0 || D_in < 0 || D_out < 0) return AWQ_ERR_SHAPE;
  if (D_in % 64 != 0 || D_in % cfg->group_size != 0 || D_out % 16 != 0) return AWQ_ERR_SHAPE;
  if (M > INT32_MAX || D_in > INT32_MAX || D_out > INT32_MAX) return AWQ_ERR_SHAPE;
  if (M == 0 || D_in == 0 || D_out == 0) return AWQ_OK;
  if (!X || !qweight || !scales || !zeros || !Y || !ws) return AWQ_ERR_INVALID_ARG;
  if (!aligned(X, 16) || !aligned(qweight, 16) || !aligned(scales, 16) || !aligned(zeros, 16) ||
      (s && !aligned(s, 16)) || !aligned(Y, 16) || !aligned(ws, 256))
    return AWQ_ERR_ALIGNMENT;
  if (ws_bytes < w4a16_ws_bytes(M, D_in, D_out)) return AWQ_ERR_WORKSPACE;
  int dev = 0;
  st = check_device(&dev);
  if (st != AWQ_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  st = get_encode(&encode);
  if (st != AWQ_OK) return st;
  if (M <= kW4a16DecodeMaxRows) {
    // a few rows: the CUDA-core path that reads the codes once
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t tb = w4a16_ticket_bytes(D_out), xb = w4a16_xprep_bytes(D_in);
    // the header and the tickets are zeroed by the path's first kernel
    uint8_t* base = static_cast<uint8_t*>(ws);
    ProfScope prof("w4a16_decode", cs);
    return from_cuda(launch_w4a16_decode(encode, X, M, D_in, D_out, qweight, scales, zeros, s, cfg->group_size, Y,
                                         reinterpret_cast<float*>(base + kHeaderBytes + tb + xb),
                                         reinterpret_cast<unsigned int*>(base + kHeaderBytes),
                                         base + kHeaderBytes + tb, status_word(ws), cs));
  }
  int pairs = 0;
  st = get_w4a16_pairs(dev, &pairs);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), cs) != cudaSuccess) return AWQ_ERR_CUDA;
  ProfScope prof("w4a16", cs);
  return from_cuda(launch_w4a16(encode, X, M, D_in, D_out, qweight, scales, zeros, s, cfg->group_size, Y,
                                status_word(ws), pairs, cs));
}

// ------------------------------------------------------------------ self-test GEMM
awq_status awq_selftest_gemm_bf16(const void* A, const void* B, int32_t b_mn_major, int64_t M, int64_t N, int64_t K,
                                  float* C, void* ws, size_t ws_bytes, awq_stream_t stream) {
  if (!A || !B || !C || !ws) return AWQ_ERR_INVALID_ARG;
  if (M < 1 || N < 8 || K < kGemmBK || K % kGemmBK != 0 || N % 8 != 0 || M > int64_t(65535) * kGemmBM ||
      K > (int64_t(1) << 30) || N > (int64_t(1) << 30))
    return AWQ_ERR_SHAPE;
  if (b_mn_major != 0 && b_mn_major != 1) return AWQ_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 4) || !aligned(ws, 256)) return AWQ_ERR_ALIGNMENT;
  if (ws_bytes < kHeaderBytes) return AWQ_ERR_WORKSPACE;
  awq_status st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  st = get_encode(&encode);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), cs) != cudaSuccess) return AWQ_ERR_CUDA;
  return from_cuda(launch_gemm_store(encode, A, B, b_mn_major, M, N, K, C, status_word(ws), cs));
}

awq_status awq_selftest_wait_timeout(uint64_t limit_ns, int32_t pairs, uint32_t* record, void* ws, size_t ws_bytes,
                                     awq_stream_t stream) {
  if (!record || !ws) return AWQ_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 2000ull * 1000ull * 1000ull) return AWQ_ERR_INVALID_ARG;
  if (pairs < 1 || pairs > 1024) return AWQ_ERR_SHAPE;
  if (!aligned(ws, 256) || !aligned(record, 4)) return AWQ_ERR_ALIGNMENT;
  if (ws_bytes < kHeaderBytes + 4096) return AWQ_ERR_WORKSPACE;
  awq_status st = check_device(nullptr);
  if (st != AWQ_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), cs) != cudaSuccess) return AWQ_ERR_CUDA;
  if (cudaMemsetAsync(record, 0, 4 * sizeof(uint32_t), cs) != cudaSuccess) return AWQ_ERR_CUDA;
  return from_cuda(launch_abort_selftest(static_cast<uint8_t*>(ws) + kHeaderBytes, limit_ns, pairs, status_word(ws),
                                         record, cs));
}

// ------------------------------------------------------------------ profiling
awq_status awq_profile_enable(int32_t enable) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.enabled = enable != 0;
  return AWQ_OK;
}

awq_status awq_profile_collect(awq_kernel_time* out, int32_t max_entries, int32_t* n_entries) {
  if (!n_entries || (max_entries > 0 && !out)) return AWQ_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  std::vector<awq_kernel_time> acc;
  awq_status st = AWQ_OK;
  for (const ProfRecord& r : g_prof.records) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      st = AWQ_ERR_CUDA;
    size_t i = 0;
    for (; i < acc.size(); ++i)
      if (r.name == acc[i].name) break;
    if (i == acc.size()) {
      awq_kernel_time t;
      std::memset(&t, 0, sizeof(t));
      std::strncpy(t.name, r.name.c_str(), sizeof(t.name) - 1);
      acc.push_back(t);
    }
    acc[i].launches += 1;
    acc[i].total_ms += ms;
    g_prof.pool.push_back(r.start);
    g_prof.pool.push_back(r.stop);
  }
  g_prof.records.clear();
  const int32_t n = static_cast<int32_t>(acc.size()) < max_entries ? static_cast<int32_t>(acc.size()) : max_entries;
  for (int32_t i = 0; i < n; ++i) out[i] = acc[i];
  *n_entries = n;
  return st;
}

}  // extern "C"
