/*
 * ggrn_timeline.h -- the profiling build of the library (libggrn_timeline.so,
 * built by `python -m gated_group_rmsnorm_gb300.build --timeline`).
 *
 * It is libggrn.so with the streaming kernels' per-CTA timeline compiled in:
 * every entry point of include/ggrn.h behaves the same, and in addition each
 * streaming launch that claims units dynamically records, per CTA, the
 * device global-timer (nanoseconds) at entry, at the release of its
 * programmatic-dependent-launch wait, when consumer warp 0 first sees a
 * stage, and at the end of its last consumer warp, plus the units it took.
 * Records are kept for 64 launches, indexed by the launch's claim epoch
 * modulo 64 (launches on the static schedule share index 0), and 320 CTAs.
 * The product path never loads this library; the benchmark's timeline mode
 * does.  No counterpart in the pages: a measurement aid.
 */
#ifndef GGRN_TIMELINE_H
#define GGRN_TIMELINE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Copy the records of the element type's kernels (bf16, f16 or f32) to
 * `host`: uint64 [64][320][5] = {entry, release, first stage, end, units};
 * 0 on success, 1 on a CUDA error.  Synchronous on the current device. */
int ggrn_timeline_read_bf16(unsigned long long* host);
int ggrn_timeline_read_f16(unsigned long long* host);
int ggrn_timeline_read_f32(unsigned long long* host);

/* Zero the records (current device); 0 on success, 1 on a CUDA error. */
int ggrn_timeline_clear_bf16(void);
int ggrn_timeline_clear_f16(void);
int ggrn_timeline_clear_f32(void);

#ifdef __cplusplus
}
#endif

#endif /* GGRN_TIMELINE_H */
