/*
 * kkt_test.h -- test hooks of libkkt.  Not part of the solve API: these entry points
 * exist so that tests can drive code paths that correct inputs never reach.
 */
#ifndef KKT_TEST_H
#define KKT_TEST_H

#include <stddef.h>
#include <stdint.h>

#include "kkt.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kkt_test_stalled_solve -- failure detection of the tensor-core kernel.
 *
 * Arguments, layouts, ownership and validation: as kkt_solve_fwd (bf16 I/O, shapes the
 * tensor-core kernel covers; others return KKT_ERR_UNSUPPORTED).  The kernel is launched
 * with the fixed round-robin schedule and with one deliberate omission: no CTA loads the
 * shared-memory stage of its first tile, so the barrier that stage would complete never
 * completes.  Every wait in the kernel is bounded (2 s), so the roles waiting on it give up,
 * record KKT_ERR_TIMEOUT in the device status word, stop the other roles of their CTA, wait
 * for their own copies and tensor-core work in flight, free tensor memory and return.  No
 * fault, trap or unbounded wait is involved and the context stays usable.
 *
 * Returns KKT_OK when the launch was made (the timeout is reported by kkt_device_status
 * after the kernel ends, about two seconds later).  The contents of T_out, W_out and U_out
 * are unspecified afterwards.
 */
int kkt_test_stalled_solve(const void *k, const void *v, const float *beta, const int32_t *cu_seqlens,
                           int B, int T, int H, int dk, int dv, int C,
                           float *T_out, void *W_out, void *U_out, struct CUstream_st *stream);

/*
 * kkt_debug_bounds -- the range checks of a bounds-checked build (library built with
 * -DKKT_DEBUG_BOUNDS, e.g. gdn_chunkwise_ut_gb300.build.build(debug_bounds=True)).
 *
 * In such a build every shared-memory access of the tensor-core kernel, every array access of
 * the SIMT kernel and every plain global load or store of both is checked against its range; a
 * failed check counts a violation and redirects the access to a scratch slot (no fault, no trap).
 * Synchronises nothing: call it after the device work has completed.  Returns the number of
 * violations since the last call and clears the records, writing the kind of the first violation
 * (1 shared memory, 2 array index, 3 global index) and its shared address or index to *kind and
 * *first (either may be NULL).  Returns -1 in the default build (no checks compiled in).
 */
int kkt_debug_bounds(unsigned long long *first, int *kind);

/*
 * kkt_test_noalloc_scratch -- copies the two 64-bit counters at the start of the scratch array
 * of kkt_solve_fwd_noalloc (current device) to out2[0..1], synchronously.  Tests use it to check
 * that every call leaves the counters zero.  Returns KKT_OK, KKT_ERR_ARG or KKT_ERR_CUDA.
 */
int kkt_test_noalloc_scratch(unsigned long long *out2);

/*
 * kkt_test_plan_pieces -- the piece plan of kkt_solve_fwd_host (host only, no CUDA call).  The
 * sequences are [starts[s], starts[s + 1]) on the flat token axis (nseq + 1 offsets); C is the chunk
 * size and parts the most pieces allowed.  Writes piece p's first row and last row + 1 to
 * bounds[2 p] and bounds[2 p + 1], the number of its sub-sequences to nsub[p], and its sub-sequence
 * offsets (relative to its first row, nsub[p] + 1 of them, the first 0) one piece after the other
 * to cu.  Returns the number of pieces, or -1 when max_pieces or cu_cap is too small or an argument
 * is invalid.
 */
int kkt_test_plan_pieces(const int64_t *starts, int nseq, int C, int parts, int64_t *bounds, int32_t *nsub,
                         int max_pieces, int32_t *cu, int cu_cap);

#ifdef __cplusplus
}
#endif

#endif /* KKT_TEST_H */
