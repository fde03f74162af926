/*
 * qmd_trace.h -- two extra entry points of the TRACED build of libqmd (libqmd_trace.so, built by
 * `python -m quantised_decode_mat_gb300.build --trace`, i.e. every kernel source compiled with
 * -DQMD_TRACE).  The product library libqmd.so does not export them.  The pages have no
 * counterpart: this is a measurement aid for the per-phase breakdown of a decode step.
 *
 * In the traced build every mat-vec (dp4a kernel) and stand-alone pack launch writes, per CTA,
 * QMD_TRACE_FIELDS = 8 unsigned 64-bit words into the next free records of a caller-owned device
 * buffer: global-timer nanoseconds at
 *   0 entry, 1 first weight copies requested, 2 dependency wait released, 3 activations ready,
 *   4 first weight stage landed, 5 the CTA's last rows written, 6 exit (the latest warp; an
 *   atomic max, so the buffer must start zeroed),
 * and word 7 = SM id | CTA index << 16 | grid << 32 | kind << 48 (kind 1 mat-vec packing its own
 * input, 2 mat-vec on packed input, 3 stand-alone pack).  The pack kernel writes 0, 2, 6 and 7.
 * A launch whose records do not fit, or any launch after qmd_debug_trace(NULL, 0), records
 * nothing.  The tensor-core kernel takes records but writes none.  Records are taken on the host
 * at launch (or at capture, for a CUDA graph, whose replays rewrite the same records).
 */
#ifndef QMD_TRACE_H
#define QMD_TRACE_H

#include <stdint.h>

#include "qmd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Use `buf` (device, 8-byte aligned, `records` x 8 words, zeroed by the caller) for the stamps of
 * the launches made after this call, from its first record on; NULL stops recording.
 * Errors: VALUE (misaligned buffer or negative count). */
qmd_status qmd_debug_trace(void *buf, int64_t records);

/* The launches recorded since the last qmd_debug_trace, in launch order: first[i] is launch i's
 * first record and ctas[i] the records it took.  Writes at most `max` entries (either pointer
 * may be NULL) and returns the number of launches recorded. */
int64_t qmd_debug_trace_launches(int64_t *first, int32_t *ctas, int64_t max);

#ifdef __cplusplus
}
#endif

#endif /* QMD_TRACE_H */
