/*
 * awq_selftest.h - test-only entry points of the B300 AWQ library.
 *
 * awq_selftest_gemm_bf16: the pages define no plain GEMM; this call exists so
 * that the tensor-core main loop used by awq_search (TMA-staged bf16 tiles,
 * tcgen05.mma into a TMEM fp32 accumulator) can be checked on its own against
 * an ordinary matrix product.  It shares the kernel template of the search
 * and differs only in the epilogue, which stores C instead of reducing
 * squares.
 *
 * awq_selftest_wait_timeout: runs the abort path that the CTA-pair kernels
 * take when a bounded wait expires, with a short limit, so that a test can
 * check its outcome without any fault.
 */
#ifndef AWQ_B300_SELFTEST_H
#define AWQ_B300_SELFTEST_H

#include "awq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* C = A * B in fp32.
 *   A  device bf16 [M, K] row-major (K contiguous)
 *   B  device bf16: b_mn_major = 1 -> [K, N] row-major (N contiguous);
 *                   b_mn_major = 0 -> [N, K] row-major (K contiguous)
 *   C  device fp32 [M, N] row-major, written
 *   ws device workspace of at least 256 bytes (status word)
 * K must be a positive multiple of 64; N a multiple of 8; pointers 16-byte
 * aligned (C 4-byte).  Asynchronous on `stream`. */
AWQ_API awq_status awq_selftest_gemm_bf16(const void* A, const void* B, int32_t b_mn_major, int64_t M, int64_t N, int64_t K,
                                  float* C, void* ws, size_t ws_bytes, awq_stream_t stream);

/* The failure path of the CTA-pair kernels, run on purpose.  (No counterpart
 * on the pages: the search and the W4A16 product bound every wait of their
 * roles on one another, and this call exercises what they do when a wait
 * expires.)
 *
 * `pairs` tcgen05 CTA pairs allocate TMEM, start a 4 KB bulk copy from
 * ws + 256 into shared memory, and then wait on mbarriers that never
 * complete, each wait bounded by limit_ns of wall time: the first wait to
 * expire records AWQ_ERR_TIMEOUT in the status word of ws and raises the
 * CTA's abort flag; the other roles leave (the epilogue-like warps agree
 * through a named barrier), the copy in flight is waited for, the two CTAs of
 * a pair meet at a cluster barrier and TMEM is freed -- the same steps and
 * helpers as the product kernels' abort path.  Nothing faults or traps; the
 * device stays usable, and the next call on ws clears the status word.
 *   limit_ns  1e3 .. 2e9 (the product kernels use 2e9)
 *   pairs     1 .. 1024
 *   record    device uint32 [4], written: [0] CTAs that freed TMEM and
 *             finished, [1] CTAs in which a wait expired, [2] the longest
 *             time a CTA ran (microseconds), [3] CTAs whose copy landed
 *             intact
 *   ws        device workspace of at least 256 + 4096 bytes, 256-byte aligned
 * After the call, awq_workspace_status(ws) returns AWQ_ERR_TIMEOUT.
 * Asynchronous on `stream`. */
AWQ_API awq_status awq_selftest_wait_timeout(uint64_t limit_ns, int32_t pairs, uint32_t* record, void* ws,
                                             size_t ws_bytes, awq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* AWQ_B300_SELFTEST_H */
