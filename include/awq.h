/*
 * awq.h - C ABI of the B300 (sm_103a) AWQ calibration hot path.
 *
 * The library computes, for one linear layer Y = X W, the steps of
 * activation-aware weight quantisation as the pages describe them:
 *
 *   1. awq_act_stats      a_j = mean_r |X[r, j]|
 *   2. awq_search         for every alpha_k of a grid: s_j = max(a_j, floor)^alpha_k,
 *                         W' = diag(s) W quantised per group of g input rows to
 *                         4 bits and dequantised, L_k = ||X S^-1 W'hat - X W||^2;
 *                         then k* = argmin_k L_k and s* = s(alpha_k*)
 *   3. awq_quantize_pack  Quantize(diag(s) W) as nibble-packed codes plus
 *                         fp16 per-group scales and zeros
 *
 * and around them: the statistic over a stream of batches and its max form
 * (awq_act_stats_accumulate / _finalize), the pack that reuses the search's
 * quantiser parameters (awq_quantize_pack_searched), the same search through
 * the Gram factor of X (awq_search_gram), the closed-form scale
 * (awq_closed_form_scales), the ADR's per-group greedy search
 * (awq_greedy_search), and the W4A16 product on the packed layer
 * (awq_w4a16_matmul).
 *
 * Sources, by page title and section:
 *   "AWQ (Activation-aware Weight Quantization)" (compassingai concept page):
 *       技术原理 - 重要通道识别的统计依据 (statistic), 缩放因子优化的完整流程
 *       steps 1-6 (grid, scaling, group quantisation, loss, argmin, s*),
 *       推理时的等效实现 (offline Quantize(diag(s*) W)), 量化数学基础 (absmax).
 *   aiqz.cc article "awq-activation-aware-quantization", sections 1, 3 and 4
 *       (E|X_i| importance; the closed-form scale; Delta = max|w_s|/7, round,
 *       clamp, dequant).
 *   "009. AWQ Integration" (ADR), Decision, 关键设计 1-3 and Consequences
 *       (add_batch statistic; per-group power-of-two greedy; search and pack
 *       share one quantiser; two 4-bit weights per byte; zeros buffer).
 *   "量化推理算法 GPTQ / AWQ" (slowleelab), L3 (H = X^T X).
 *   CSDN AutoAWQ deployment walkthrough, section 2 (quant_config:
 *       zero_point, q_group_size 128, w_bit 4).
 *
 * Conventions shared by every call
 *   - All matrices are row-major with a contiguous inner dimension.
 *     X is [N, D_in] bf16 (N calibration rows), W is [D_in, D_out] bf16
 *     (input channel j = row j; groups run down the rows).
 *   - Device pointers must be 16-byte aligned; D_in and D_out must be
 *     multiples of 8.
 *   - The caller owns every buffer, including the workspace `ws`; the library
 *     allocates no device memory and keeps no state between calls (other than
 *     a per-device cache of the architecture check and driver entry points).
 *   - Every compute call is asynchronous on `stream` (NULL = legacy default
 *     stream): it validates its arguments on the host, enqueues its kernels
 *     and returns.  A host-side validation failure returns an error before
 *     anything is enqueued and before any CUDA call is made.
 *   - Errors found on the device (a quantisation step that overflows fp16, a
 *     non-finite input, a bounded wait that expired) are written to a status
 *     word at the start of `ws`; each call clears that word first.  Read it
 *     with awq_workspace_status(), which synchronises `stream`.
 *   - Only sm_103 devices are supported; any other device makes a call
 *     return AWQ_ERR_UNSUPPORTED_DEVICE.  There is no fallback path.
 */
#ifndef AWQ_B300_AWQ_H
#define AWQ_B300_AWQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define AWQ_API __attribute__((visibility("default")))
#else
#define AWQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same handle type); NULL selects the legacy default stream. */
typedef struct CUstream_st* awq_stream_t;

typedef enum {
  AWQ_OK = 0,
  AWQ_ERR_INVALID_ARG = 1,         /* null pointer, bad cfg field or grid value      */
  AWQ_ERR_SHAPE = 2,               /* sizes out of range or not divisible             */
  AWQ_ERR_ALIGNMENT = 3,           /* pointer not 16-byte aligned                     */
  AWQ_ERR_WORKSPACE = 4,           /* workspace smaller than the size query returned  */
  AWQ_ERR_UNSUPPORTED_DEVICE = 5,  /* current device is not sm_103                    */
  AWQ_ERR_CUDA = 6,                /* a CUDA runtime/driver call failed               */
  AWQ_ERR_RANGE = 7,               /* a quantisation step does not fit in fp16        */
  AWQ_ERR_NONFINITE = 8,           /* NaN or infinity in an input                     */
  AWQ_ERR_TIMEOUT = 9              /* a bounded device wait expired (kernel returned) */
} awq_status;

/* Quantiser configuration (the pages' quant_config: w_bit, q_group_size, zero_point). */
typedef struct {
  int32_t bits;        /* must be 4                                                     */
  int32_t group_size;  /* 64, 128 or 256 input rows per group; must divide D_in         */
  int32_t symmetric;   /* 0: asymmetric min-max with a zero point; 1: absmax, codes -7..7 */
  float act_floor;     /* lower clamp of the statistic before the power (1e-4)          */
} awq_cfg;

/* Human-readable name of a status code (static string, never NULL). */
AWQ_API const char* awq_status_string(awq_status status);

/* Synchronises `stream` and returns the status word a previous call on the
 * same workspace left on the device (AWQ_OK if no device error was seen). */
AWQ_API awq_status awq_workspace_status(const void* ws, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Step 1: per-input-channel activation statistic.
 * "AWQ (Activation-aware Weight Quantization)", 技术原理 - 重要通道识别的统计依据:
 * activation_scale[j] = mean(|X_calib[:, j]|); aiqz.cc article section 1,
 * I_i = E[|X_i|].
 *
 *   X        device, bf16 [N, D_in], row stride ldx elements (ldx >= D_in, ldx % 8 == 0)
 *   mean_abs device, fp32 [D_in], written: (1/N) sum_r |X[r, j]|
 *   ws       device workspace of at least awq_act_stats_workspace_size() bytes
 * N must be >= 1 (a mean over no rows is undefined: AWQ_ERR_SHAPE); D_in == 0
 * is a no-op.  Sums are fp32 within a row slice and fp64 across slices, in a
 * fixed order, so the result is deterministic.  A non-finite X sets
 * AWQ_ERR_NONFINITE in the workspace status.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_act_stats_workspace_size(int64_t N, int64_t D_in, size_t* bytes);
AWQ_API awq_status awq_act_stats(const void* X, int64_t N, int64_t D_in, int64_t ldx,
                         float* mean_abs, void* ws, size_t ws_bytes, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The statistic over a stream of calibration batches, and its max variant.
 *
 * "009. AWQ Integration", Decision (Layer 2): the quantizer's add_batch
 * accumulates the per-channel mean |x| batch by batch; "AWQ (Activation-aware
 * Weight Quantization)", 二、缩放因子的搜索 / 重要通道识别的统计依据: the
 * statistic may also be max |X_j| ("或 max"), s_j = (max |X_j|)^alpha.
 *
 * awq_act_stats_accumulate adds one batch:
 *   X, N, D_in, ldx   the batch, as for awq_act_stats (N >= 1 rows)
 *   sum_abs  device, fp64 [D_in], read and written: sum_abs[j] += sum_r |X[r, j]|
 *            (the batch's sum formed in the same fixed order as awq_act_stats)
 *   max_abs  device, fp32 [D_in] or NULL: max_abs[j] = max(max_abs[j], max_r |X[r, j]|)
 *   ws       as for awq_act_stats
 * The caller zeroes sum_abs and max_abs before the first batch and orders the
 * batches on one stream.  awq_act_stats_finalize writes mean_abs[j] =
 * fp32(sum_abs[j] / rows) for rows = the total number of rows accumulated.
 * Either vector (mean or max) can then be passed to awq_search as its
 * statistic.  A non-finite batch sets AWQ_ERR_NONFINITE in ws.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_act_stats_accumulate(const void* X, int64_t N, int64_t D_in, int64_t ldx, double* sum_abs,
                                            float* max_abs, void* ws, size_t ws_bytes, awq_stream_t stream);
AWQ_API awq_status awq_act_stats_finalize(const double* sum_abs, int64_t rows, int64_t D_in, float* mean_abs,
                                          awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The same statistic for callers that cannot allocate device memory.
 * (No counterpart on the pages: this is a library convenience.)
 *
 * Some callers have no way to obtain a workspace: a plug-in running inside a
 * host program that has already reserved all device memory for its own pool
 * and exposes no allocator, or code on a latency-critical path that must not
 * call cudaMalloc (which can synchronise the whole device).  This entry point
 * takes only X and the output; its scratch (a status word, one completion
 * counter per 256 channels and the per-row-slice partial sums) is a
 * 256 B + 16 KiB + 4 MiB array of static device memory inside the library,
 * which every device that loads the library holds until the process exits.
 * Each call clears the status word and the counters it uses
 * (cudaMemsetAsync on the array, which allocates nothing).
 *
 *   X, N, D_in, ldx, mean_abs  as for awq_act_stats
 * Limits: D_in <= 1048576 channels; larger D_in returns AWQ_ERR_SHAPE without
 * launching anything.  The call makes no cudaMalloc / cudaFree and uses no
 * allocating library routine.  The first call on a device looks up the
 * array's device address for that device (cudaGetSymbolAddress, with that
 * device current); make that first call before any stream capture.  The
 * address is kept per device and CUDA context: after cudaDeviceReset the next
 * call looks it up again in the new context (again a first call, to be made
 * outside a capture).  Every call shares the one array: calls whose kernels
 * overlap on the GPU (e.g. on two streams) race and corrupt each other's
 * result, so serialise them.  Results are bit-identical to awq_act_stats'
 * (same row-slice plan, same kernel, same summation order).  There is no
 * status word for the caller to read, so device-side failures show up in the
 * output: a non-finite X gives a non-finite entry of mean_abs, and a bounded
 * device wait that expires (AWQ_ERR_TIMEOUT in the other entry points) makes
 * the means of the affected 256-channel chunk NaN.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_act_stats_noalloc(const void* X, int64_t N, int64_t D_in, int64_t ldx,
                                         float* mean_abs, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Steps 2-3: the alpha-grid scale search and its argmin.
 * "AWQ (Activation-aware Weight Quantization)", 缩放因子优化的完整流程 steps 3-6:
 * s_j(alpha) = activation_scale[j]^alpha, W' = diag(s) W, W4 per-group
 * quantisation, L(alpha) = ||X S^-1 W'hat - X W||^2, alpha* = argmin, s*.
 *
 *   X          device, bf16 [N, D_in] contiguous
 *   W          device, bf16 [D_in, D_out] contiguous
 *   mean_abs   device, fp32 [D_in] (the output of awq_act_stats)
 *   grid       HOST, fp64 [G] exponents alpha_k in [0, 1] (the pages use k/20, G = 21)
 *   G          1 <= G <= 64
 *   losses     device, fp64 [G], written: L_k (plain sum of squares)
 *   best_idx   device, int32 [1], written: first k with the smallest L_k
 *   s_star     device, fp32 [D_in], written: s(alpha_best)
 *   col_losses device, fp64 [G, D_out] or NULL; if given, written with the
 *              per-output-column share of L_k (L_k = sum_n col_losses[k, n])
 *   ws         device workspace of at least awq_search_workspace_size() bytes
 * Scales are s_j = (float)pow((double)max(mean_abs[j], act_floor), alpha_k).
 * Candidate losses use bf16 tensor-core products with fp32 accumulation and
 * an fp64 fixed-order reduction; results are deterministic run to run.
 * N >= 1; D_in a multiple of group_size; D_out a multiple of 8.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_search_workspace_size(int64_t N, int64_t D_in, int64_t D_out, int32_t G,
                                     const awq_cfg* cfg, size_t* bytes);
AWQ_API awq_status awq_search(const void* X, const void* W, int64_t N, int64_t D_in, int64_t D_out,
                      const float* mean_abs, const double* grid, int32_t G, const awq_cfg* cfg,
                      double* losses, int32_t* best_idx, float* s_star, double* col_losses,
                      void* ws, size_t ws_bytes, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The search sharded over output columns (several processes, one GPU each).
 * "AWQ (Activation-aware Weight Quantization)", 缩放因子优化的完整流程 step 4c:
 * L is a squared Frobenius norm, a sum over output columns, so the candidates'
 * losses of the whole layer are the sums of the losses of disjoint column
 * slices.  Each rank runs awq_search on X and its slice W[:, c0:c1], copies
 * out the search's block partials, the ranks gather them in slice order, and
 * each rank selects the global alpha* from all of them; the searched pack of
 * each slice then uses that alpha*.
 *
 * awq_search_block_losses: after awq_search(N, D_in, D_out, G, cfg, ws), its
 *   fp64 block partials: blk [G, nb], nb = ceil(D_out / 256); blk[k][b] is
 *   the candidate-k loss of columns [256 b, 256 b + 256), summed in the
 *   search's fixed order.  Device to device copy, asynchronous on `stream`.
 * awq_search_select: blk holds [G, nb] block partials of all slices, each
 *   slice's blocks in column order and the slices in order (nb the total);
 *   writes losses [G] (the blocks summed in order, fp64), best_idx (first
 *   smallest loss) and s_star [D_in] (s of that candidate, from the scale
 *   table in ws), into the caller's buffers.  ws, N, D_in, D_out, G, cfg: this
 *   rank's own awq_search call; pass that call's losses, best_idx and s_star
 *   to overwrite them, so that awq_quantize_pack_searched on ws packs this
 *   rank's slice at the global alpha*.  When every slice but the last spans a
 *   multiple of 256 columns, the losses equal those of one awq_search of the
 *   whole layer bit for bit.  All losses NaN: AWQ_ERR_NONFINITE in ws.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_search_block_losses(const void* ws, size_t ws_bytes, int64_t N, int64_t D_in, int64_t D_out,
                                           int32_t G, const awq_cfg* cfg, double* blk, awq_stream_t stream);
AWQ_API awq_status awq_search_select(const double* blk, int64_t nb, int32_t G, void* ws, size_t ws_bytes,
                                     int64_t N, int64_t D_in, int64_t D_out, const awq_cfg* cfg, double* losses,
                                     int32_t* best_idx, float* s_star, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Step 4: offline quantisation and nibble packing of diag(s) W.
 * "AWQ (Activation-aware Weight Quantization)", 推理时的等效实现:
 * W_quantized = Quantize(diag(s*) W); "009. AWQ Integration", Consequences:
 * two 4-bit weights per byte.
 *
 *   W        device, bf16 [D_in, D_out] contiguous
 *   s        device, fp32 [D_in] per-input-channel scale (normally s_star)
 *   qweight  device, uint8 [D_in/2, D_out]: byte (i, n) = code(2i, n) | code(2i+1, n) << 4
 *   scales   device, fp16 [D_in/group_size, D_out]: quantisation step per (group, column)
 *   zeros    device, fp16 [D_in/group_size, D_out]: zero point per (group, column)
 * Dequantisation is (code - zero) * scale, then / s_j for the original weight.
 * Asymmetric: step = fp16((max(w',0) - min(w',0)) / 15), zero = clamp(rint(-min/step), 0, 15),
 *             code = clamp(rint(w'/step) + zero, 0, 15).
 * Symmetric:  step = fp16(max|w'| / 7), code = clamp(rint(w'/step), -7, 7) + 8, zero = 8.
 * Divisions are IEEE fp32 round-to-nearest and rint rounds half to even, so
 * codes, scales and zeros are exact functions of (W, s).  A zero step gives
 * code 0 (asymmetric, zero 0) or 8 (symmetric).  A step above the fp16 range
 * sets AWQ_ERR_RANGE; a non-finite W sets AWQ_ERR_NONFINITE.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_pack_workspace_size(int64_t D_in, int64_t D_out, const awq_cfg* cfg, size_t* bytes);
AWQ_API awq_status awq_quantize_pack(const void* W, const float* s, int64_t D_in, int64_t D_out,
                             const awq_cfg* cfg, uint8_t* qweight, void* scales, void* zeros,
                             void* ws, size_t ws_bytes, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The same search through the Gram matrix of X (N >= D_in).
 *
 * Every candidate's loss is a quadratic form in H = X^T X:
 *     L_k = ||X D_k||^2 = sum_n d_n^T H d_n,   D_k = S_k^-1 W'hat_k - W,
 * so with the Cholesky factor H = L L^T the search can run on R = L^T
 * (D_in rows) in place of X (N rows): 2 D_in^2 D_out flops per candidate
 * instead of 2 N D_in D_out, after one 2 N D_in^2 product for H and
 * D_in^3 / 3 for the factor.  Worth it when N is well above D_in.
 *
 * Arguments, outputs and conventions as for awq_search; ws of
 * awq_search_gram_workspace_size() bytes, which begins with a search
 * workspace, so awq_quantize_pack_searched(search_ws = ws) works after it.
 * H is accumulated in fp32 from the bf16 X on the tensor cores, factored in
 * fp32 (64 x 64 blocks) and R rounded to bf16, so the losses differ from
 * awq_search's by the rounding of R (well inside the 1e-2 loss tolerance on
 * the test layers).  A factor that is not positive definite (rank-deficient
 * X) sets AWQ_ERR_RANGE.  Requires N >= D_in and D_in a multiple of 64.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_search_gram_workspace_size(int64_t N, int64_t D_in, int64_t D_out, int32_t G,
                                                  const awq_cfg* cfg, size_t* bytes);
AWQ_API awq_status awq_search_gram(const void* X, const void* W, int64_t N, int64_t D_in, int64_t D_out,
                                   const float* mean_abs, const double* grid, int32_t G, const awq_cfg* cfg,
                                   double* losses, int32_t* best_idx, float* s_star, double* col_losses, void* ws,
                                   size_t ws_bytes, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Step 4 right after a search: the same packing, with the per-group
 * quantiser parameters the search already computed for its best candidate.
 *
 * awq_search evaluates every candidate with the pack's own quantiser (adr
 * "009. AWQ Integration", 关键设计 3: search and pack share one quantiser), so
 * its workspace already holds, for alpha*, the exact step (fp16-rounded) and
 * zero of every (group, column) that awq_quantize_pack would compute from
 * diag(s*) W.  This call reads them instead of recomputing them and packs in
 * one streaming pass over W.
 *
 *   W, D_in, D_out, cfg    the same W and cfg as the awq_search call
 *   G                      that call's grid size
 *   search_ws, search_ws_bytes  that call's workspace, unchanged since
 *   best_idx, s_star       that call's device outputs (s_star 16-byte aligned)
 *   qweight, scales, zeros as for awq_quantize_pack (scales, zeros 16-byte aligned)
 * The outputs equal awq_quantize_pack(W, s_star, ...) bit for bit.  Device
 * errors of W (non-finite values, fp16 step overflow) were already reported
 * in the search workspace's status word; this call adds none.  Must be
 * ordered after the search on the device (same stream, or an event).
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_quantize_pack_searched(const void* W, int64_t D_in, int64_t D_out, int32_t G,
                                              const awq_cfg* cfg, const void* search_ws, size_t search_ws_bytes,
                                              const int32_t* best_idx, const float* s_star, uint8_t* qweight,
                                              void* scales, void* zeros, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The closed-form scale (aiqz.cc article "awq-activation-aware-quantization",
 * section 3): one scale per input channel without a search,
 *     s_i = (E|X_i|)^alpha / mean_j |W_ij|,   alpha in [0, 1] (0.5 by default).
 *
 *   W, D_in, D_out   device, bf16 [D_in, D_out] (D_out a multiple of 8); row i = channel i
 *   mean_abs         device, fp32 [D_in]: E|X_i| (awq_act_stats), floored at cfg->act_floor
 *   s_out            device, fp32 [D_in], written
 * mean_j |W_ij| is summed in fp64 (exact for rows spanning up to ~30
 * binades), the quotient formed in fp64 and rounded once to fp32; a row of
 * zeros gets s = 1.  s_out can be passed to awq_quantize_pack.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_closed_form_scales(const void* W, int64_t D_in, int64_t D_out, const float* mean_abs,
                                          double alpha, const awq_cfg* cfg, float* s_out, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * The ADR's second search: per-group coordinate greedy over power-of-two
 * channel scales ("009. AWQ Integration", 关键设计 1-3).
 *
 * Groups of cfg->group_size input rows are independent.  Starting from
 * s = 1, for each pass and each channel j of a group in index order, every
 * candidate 2^k (k = k_min .. k_min + n_cand - 1) is tried for s_j with the
 * group's other scales fixed, and the group's activation-weighted
 * reconstruction error
 *     E = sum_i a_i sum_n (w'hat_in / s_i - w_in)^2,  w' = w s,
 * is evaluated with the pack's own quantiser (cfg); s_j moves to the best
 * candidate when that is strictly better than its current value (the first
 * in k order among equals).  The ADR's defaults: passes 3, 20 candidates
 * centred on 1 (k_min = -10).
 *
 *   W, D_in, D_out   device, bf16 [D_in, D_out] (D_in a multiple of group_size, D_out of 8)
 *   mean_abs         device, fp32 [D_in]: the channel weights a_i (awq_act_stats)
 *   s_out            device, fp32 [D_in], written: the final scales (powers of two)
 *   trace            device, int32 [passes, D_in] or NULL: the candidate index chosen at each step
 *   errors           device, fp64 [passes, D_in, n_cand] or NULL: E of every candidate at each step
 *   ws               device workspace of awq_greedy_workspace_size() bytes
 * Per-column errors are fp32; a group's candidates are compared on their
 * error changes against the part common to all of them, summed in a fixed
 * order in fp64, so the result is deterministic.  Constraints: 1 <= passes
 * <= 16, 1 <= n_cand <= 24, 1 among the candidates.  s_out can be passed to
 * awq_quantize_pack.  A step above the fp16 range sets AWQ_ERR_RANGE in ws.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_greedy_workspace_size(int64_t D_in, int64_t D_out, const awq_cfg* cfg, size_t* bytes);
AWQ_API awq_status awq_greedy_search(const void* W, const float* mean_abs, int64_t D_in, int64_t D_out,
                                     const awq_cfg* cfg, int32_t passes, int32_t k_min, int32_t n_cand, float* s_out,
                                     int32_t* trace, double* errors, void* ws, size_t ws_bytes, awq_stream_t stream);

/* ---------------------------------------------------------------------------
 * After the path: the W4A16 product on the packed layer.
 *
 * "AWQ (Activation-aware Weight Quantization)", 推理时的等效实现: the layer is
 * stored as W_quantized = Quantize(diag(s*) W) with s* as metadata, and at
 * inference Y = (X diag(1/s*)) Dequant(W_quantized), the 1/s* scaling folded
 * into the kernel's dequantisation (the pipeline figure's "Dequant + MatMul
 * (融合 s* 缩放)"); Dequant = (code - zero) * scale per group.
 *
 *   X        device, bf16 [M, D_in] contiguous (the layer's input activations)
 *   qweight, scales, zeros   device, the outputs of awq_quantize_pack (or
 *            awq_quantize_pack_searched) for this layer and cfg->group_size
 *   s        device, fp32 [D_in]: the s* the layer was packed with, or NULL
 *            for the plain product X Dequant(qweight)
 *   Y        device, bf16 [M, D_out] contiguous (written)
 *   ws       device workspace of awq_w4a16_workspace_size(M, D_in, D_out) bytes
 * M > 4 (prefill): each weight enters the tensor cores as bf16(((code -
 * zero) * scale) * RN(1/s_j)) and the products accumulate in fp32.  M <= 4
 * (decode): each code is read once and enters the tensor cores as the exact
 * bf16 value 128 + code, against x' = fp32(x / s) split into bf16 hi + lo
 * parts; per group the kernel forms scale * (D - (zero + 128) * sum_j x'_j)
 * with fp32 sums, and adds the per-CTA segments in a fixed order (fp32
 * trees of 8).  Y is rounded to bf16.  The decode form writes the workspace
 * header and its ticket counters itself (its first kernel zeroes them), and
 * its product kernel may begin before that kernel ends (programmatic
 * dependent launch; nothing it reads from the first kernel is read before
 * it waits for it).  Shapes: D_in a multiple of 64 and of group_size, D_out a multiple
 * of 16; all pointers 16-byte aligned (ws 256).  M = 0 is a no-op.  A
 * timeout of the kernel's bounded waits sets AWQ_ERR_TIMEOUT in the status
 * word.
 * ------------------------------------------------------------------------- */
AWQ_API awq_status awq_w4a16_workspace_size(int64_t M, int64_t D_in, int64_t D_out, size_t* bytes);
AWQ_API awq_status awq_w4a16_matmul(const void* X, int64_t M, int64_t D_in, int64_t D_out, const uint8_t* qweight,
                                    const void* scales, const void* zeros, const float* s, const awq_cfg* cfg,
                                    void* Y, void* ws, size_t ws_bytes, awq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* AWQ_B300_AWQ_H */
