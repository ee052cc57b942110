/*
 * awq_selftest.h - test-only entry point of the B300 AWQ library.
 *
 * The pages define no plain GEMM; this call exists so that the tensor-core
 * main loop used by awq_search (TMA-staged bf16 tiles, tcgen05.mma into a
 * TMEM fp32 accumulator) can be checked on its own against an ordinary
 * matrix product.  It shares the kernel template of the search and differs
 * only in the epilogue, which stores C instead of reducing squares.
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

#ifdef __cplusplus
}
#endif
#endif /* AWQ_B300_SELFTEST_H */
