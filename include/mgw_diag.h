/* mgw_diag.h -- entry points of the diagnostic library libmgw_diag.so.
 *
 * libmgw_diag.so is libmgw.so with its wgrad (CTA-pair) and fp32 dgrad kernels compiled with
 * diagnostics; it exports every function of mgw.h plus the two below, which libmgw.so does
 * not export.  The diagnostics:
 *   - a work-item timeline: per CTA and work item, the globaltimer (ns) when the item's
 *     epilogue began waiting for its accumulator and when the item's results had been
 *     stored, and the SM that ran it (the post-attn page stamps a per-CTA timeline behind a
 *     compile-time flag; this is the same tool for these kernels);
 *   - device bounds checks on the global addresses the kernels compute: a store outside its
 *     output tensor is skipped and a TMA load outside its tensor is reported (TMA fills the
 *     outside with zeros); both OR MGW_DEV_BOUNDS (mgw.h) into the call's status word.
 * The results are the same as libmgw.so's; the kernels run a little slower.  The timeline
 * buffers are device globals of the library: calls on several streams at once append to the
 * same buffers.
 */
#ifndef MGW_DIAG_H
#define MGW_DIAG_H

#include <stdint.h>

#include "mgw.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MGW_DIAG_KERNEL_WGRAD_PAIR 1 /* grouped_wgrad_pair_kernel: item = (expert, tile) index */
#define MGW_DIAG_KERNEL_DGRAD 2      /* grouped_dgrad_kernel: item = (expert, row tile, k tile) */
#define MGW_DIAG_KERNEL_DGRAD_PAIR 3 /* grouped_dgrad_pair_kernel: item = (expert, pair tile, k tile) */

typedef struct mgw_diag_record {
  uint32_t kernel;    /* MGW_DIAG_KERNEL_* */
  uint32_t sm;        /* SM id (%smid) of the CTA */
  uint32_t cta;       /* blockIdx.x */
  uint32_t reserved;
  int64_t item;       /* the kernel's work-item index */
  uint64_t t_wait_ns; /* globaltimer: the epilogue starts waiting for the item's accumulator */
  uint64_t t_done_ns; /* globaltimer: the item's stores are issued */
} mgw_diag_record;

/* Copies up to `cap` records of the timeline since the last reset to host memory `out`
 * (the wgrad records first, then the dgrad, then the CTA-pair dgrad ones) and sets *total to
 * the number recorded, which may exceed what was copied (each kernel family keeps at most
 * 65536).  Synchronises with the device (cudaMemcpyFromSymbol).  MGW_ERR_INVALID_ARG for a
 * null `out` with cap > 0 or a null `total`. */
mgw_status mgw_diag_timeline(mgw_diag_record *out, int cap, int *total);

/* Empties the timeline (all kernel families). */
mgw_status mgw_diag_timeline_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* MGW_DIAG_H */
