/*
 * awq_profile.h - optional per-kernel timing of the B300 AWQ library.
 *
 * Not part of the method the pages describe: a measurement aid.  While
 * enabled, every kernel launch made by the library is bracketed by two CUDA
 * events recorded on the launch stream; awq_profile_collect() synchronises
 * those events and returns per-kernel totals.  Disabled by default; the
 * events are created on first use and kept for reuse.
 */
#ifndef AWQ_B300_PROFILE_H
#define AWQ_B300_PROFILE_H

#include "awq.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  char name[48];       /* kernel name, e.g. "search_gemm"              */
  int64_t launches;    /* launches timed since the last collect         */
  double total_ms;     /* summed event-to-event time of those launches  */
} awq_kernel_time;

/* Enable (1) or disable (0) event timing of subsequent launches (process-wide). */
AWQ_API awq_status awq_profile_enable(int32_t enable);

/* Synchronise the recorded events and write up to `max_entries` per-kernel
 * totals into `out` (names in first-launch order); *n_entries receives the
 * count.  Clears the accumulated records. */
AWQ_API awq_status awq_profile_collect(awq_kernel_time* out, int32_t max_entries, int32_t* n_entries);

#ifdef __cplusplus
}
#endif
#endif /* AWQ_B300_PROFILE_H */
