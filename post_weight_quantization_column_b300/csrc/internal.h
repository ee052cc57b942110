// Internal launch interface between the C-ABI layer and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "status.h"

namespace awqdev {

// ----------------------------------------------------------------- stats
constexpr int kStatsRowLanes = 8;      // consumer warps per CTA, each on its own rows of a box
constexpr int kStatsThreads = (kStatsRowLanes + 1) * 32;  // + one producer warp
constexpr int kStatsCols = 256;        // channels per CTA (32 lanes x 8)
constexpr int kStatsBoxRows = 32;      // rows per ring stage (one tensor copy per box)
constexpr int kStatsStages = 6;        // ring depth: 6 x 16 KB
constexpr int kStatsTargetCtas = 148 * 2;  // two CTAs (2 x 105 KB shared memory) on each SM
constexpr int kStatsMaxSplits = 1024;

void stats_plan(int64_t N, int64_t D, int* splits, int64_t* rows_per_split);
// Column chunks of 256 channels: the number of ticket counters the kernel uses.
int64_t stats_chunks(int64_t D);
// partial: fp32 [splits][D] scratch; tickets: uint32 [stats_chunks(D)], zero on
// entry (the kernel leaves them zero again).  nan_on_error: means of a chunk
// are written as NaN when the status word is non-zero once its slices are in
// (for a status word the caller never reads).
cudaError_t launch_act_stats(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, int64_t N, int64_t D,
                             int64_t ldx, float* mean_abs, double* sum_abs, float* max_abs, float* partial,
                             float* partial_max, unsigned int* tickets, int splits, int64_t rows_per_split,
                             uint32_t* status, int nan_on_error, cudaStream_t stream);
cudaError_t launch_stats_finalize(const double* sum_abs, int64_t rows, int64_t D, float* mean_abs,
                                  cudaStream_t stream);
// The driver's tensor-map encoder (resolved once per process).
awq_status tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn);

// ----------------------------------------------------------------- quantiser
constexpr int kMaxGrid = 64;
struct AlphaGrid {
  double a[kMaxGrid];
};

// Quantiser parameters of one (candidate, group, column) used by the search:
//   inv = 1/step (0 for a zero step), zm = 1.5*2^23 + zero, step.
struct QParam {
  float inv, zm, step, pad;
};
// In memory they are stored per (candidate, group) in chunks of 8 output
// columns: {inv x8, zm x8, step x8, clamp, 3 unused} = 28 floats (112 bytes).
// clamp is 1.0 when some code of the chunk's 8 columns would leave the code
// range without the clamps (else 0.0), so readers may drop them.  The
// 112-byte stride spreads the 8 chunks read by 8 neighbouring producer
// threads over all 32 shared-memory banks.
constexpr int kQChunkCols = 8;
constexpr int kQChunkFloats = 28;
constexpr int kQChunkClamp = 3 * kQChunkCols;  // float index of the chunk's clamp flag
inline size_t qparam_floats(int G, int64_t T, int64_t D_out) {
  return static_cast<size_t>(G) * static_cast<size_t>(T) * static_cast<size_t>(D_out / kQChunkCols) * kQChunkFloats;
}

cudaError_t launch_scale_table(const float* mean_abs, int64_t D_in, const AlphaGrid& grid, int G, float act_floor,
                               float* s_tab, float* r_tab, uint32_t* status, cudaStream_t stream);
// s_i = (max(a_i, floor))^alpha / mean_j |W_ij| (a zero row: 1).
cudaError_t launch_closed_form(const void* W, int64_t D_in, int64_t D_out, const float* mean_abs, double alpha,
                               float act_floor, float* s_out, cudaStream_t stream);
cudaError_t launch_group_params(const void* W, const float* s_tab, int64_t D_in, int64_t D_out, int G,
                                int group_size, int symmetric, float* qp, uint32_t* status, cudaStream_t stream);
cudaError_t launch_pack(const void* W, const float* s, int64_t D_in, int64_t D_out, int group_size, int symmetric,
                        uint8_t* qweight, void* scales, void* zeros, uint32_t* status, cudaStream_t stream);
// Pack with the group parameters a search computed for its best candidate
// (qp: the search workspace's parameter table, best_idx: device int32).
cudaError_t launch_pack_searched(const void* W, const float* s, const float* qp, const int32_t* best_idx, int G,
                                 int64_t D_in, int64_t D_out, int group_size, int symmetric, uint8_t* qweight,
                                 void* scales, void* zeros, cudaStream_t stream);

// ----------------------------------------------------------------- tensor-core self-test
constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;

// Plain C = A * B in fp32 through a tcgen05 main loop (TMA ring, TMEM
// accumulator): the self-test of the UMMA descriptors the search relies on.
cudaError_t launch_gemm_store(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* A, const void* B, int b_mn_major,
                              int64_t M, int64_t N, int64_t K, float* C, uint32_t* status, cudaStream_t stream);

// Test-only: `pairs` CTA pairs run the abort protocol of the pair kernels on
// mbarriers that never complete, with waits bounded by limit_ns (src: 4 KB of
// device memory, 16-byte aligned, copied into each CTA; record: uint32 [4]).
cudaError_t launch_abort_selftest(const void* src, uint64_t limit_ns, int pairs, uint32_t* status, uint32_t* record,
                                  cudaStream_t stream);

// ----------------------------------------------------------------- fused search (CTA pairs)
// Rows of X per partial-sum slot of the fused search: [G][m_tiles][D_out].
int search_fused_m_tiles(int64_t N);
// CTA pairs that fit on the device at once (occupancy query).
cudaError_t search_fused_max_pairs(int* pairs);
// Decode-sized W4A16 product (M <= kW4a16DecodeMaxRows): the B fragments of
// x' = x / s into xf [xprep bytes], then a persistent register-fed MMA kernel.
constexpr int64_t kW4a16DecodeMaxRows = 4;
int64_t w4a16_decode_partial_floats(int64_t M, int64_t D_in, int64_t D_out);
int64_t w4a16_decode_tickets(int64_t D_out);
int64_t w4a16_decode_xprep_bytes(int64_t D_in);
cudaError_t launch_w4a16_decode(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, int64_t M, int64_t D_in,
                                int64_t D_out, const uint8_t* qweight, const void* scales, const void* zeros,
                                const float* s, int group_size, void* Y, float* partial, unsigned int* tickets,
                                uint8_t* xf, uint32_t* status, cudaStream_t stream);
// The Gram form of the search: X^T (zero past N, row length ldt), the
// blocked fp32 Cholesky of H in place (lower; Linv: a 64 x 64 fp32 scratch
// block), R = L^T in bf16.
cudaError_t launch_transpose_x(const void* X, int64_t N, int64_t D, int64_t ldt, void* Xt, cudaStream_t stream);
cudaError_t launch_cholesky(float* A, int64_t D, float* Linv, uint32_t* status, cudaStream_t stream);
cudaError_t launch_lt_to_bf16(const float* L, int64_t D, void* R, cudaStream_t stream);
// The adr's per-group coordinate greedy over power-of-two scales 2^k,
// k = k_min .. k_min + ncand - 1 (ncand <= kMaxGreedyCand).
constexpr int kMaxGreedyCand = 24;
int64_t greedy_slices(int64_t D_out);
cudaError_t launch_greedy(const void* W, const float* a, int64_t D_in, int64_t D_out, int group_size, int symmetric,
                          int passes, int k_min, int ncand, float* s_cur, int* cur_idx, float* partial,
                          unsigned int* tickets, int* trace, double* errors, uint32_t* status, cudaStream_t stream);
// W4A16 product Y = (X diag(1/s)) Dequant(qweight) on CTA pairs (s may be null).
cudaError_t w4a16_max_pairs(int* pairs);
cudaError_t launch_w4a16(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, int64_t M, int64_t D_in,
                         int64_t D_out, const uint8_t* qweight, const void* scales, const void* zeros, const float* s,
                         int group_size, void* Y, uint32_t* status, int max_pairs, cudaStream_t stream);
cudaError_t launch_search_fused(PFN_cuTensorMapEncodeTiled_v12000 encode, const void* X, const void* W,
                                const float* s_tab, const float* r_tab, const float* qp, int64_t N, int64_t D_in,
                                int64_t D_out, int G, int group_size, int symmetric, float* partial,
                                uint32_t* status, int max_pairs, cudaStream_t stream);

// ----------------------------------------------------------------- reductions
int reduce_blocks(int64_t D_out);
constexpr int kReduceBlockCols = 256;  // columns summed by one block partial
// L_k = the blocks of blk [G][nb] summed in order, first argmin, s* = s_k*.
cudaError_t launch_select_losses(const double* blk, int64_t nb, int G, double* losses, int32_t* best_idx,
                                 const float* s_tab, int64_t D_in, float* s_star, uint32_t* status,
                                 cudaStream_t stream);
// blk: fp64 [G][reduce_blocks(D_out)] scratch; ticket: a zeroed uint32 (left zeroed).
cudaError_t launch_reduce_losses(const float* partial, int m_tiles, int64_t D_out, int G, double* col_losses,
                                 double* blk, unsigned int* ticket, double* losses, int32_t* best_idx,
                                 const float* s_tab, int64_t D_in, float* s_star, uint32_t* status,
                                 cudaStream_t stream);

}  // namespace awqdev
