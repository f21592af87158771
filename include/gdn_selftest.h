/*
 * gdn_selftest.h -- device self-test of the bounded waits in libgdn.
 *
 * Every pipelined kernel of the library hands work between its warp roles
 * through mbarrier phases and release/acquire counters, and every such wait
 * is bounded: after GDN_OPT_WAIT_LIMIT suspending polls it gives up, marks its
 * CTA as aborting and records a timeout in the device error word, which
 * gdn_sync_check() turns into GDN_ERR_DEVICE_TIMEOUT.  The pages describe no
 * such mechanism (no paper counterpart): it is the library's own failure
 * detection, and this entry point exercises it without any fault.
 */
#ifndef GDN_SELFTEST_H
#define GDN_SELFTEST_H

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Runs one CTA that waits, through the same bounded-wait code as the
 * pipelined kernels, first on an mbarrier phase and then on a shared-memory
 * counter.
 *   complete    1: the CTA completes the phase and sets the counter before
 *               waiting, so both waits succeed and no error is recorded;
 *               0: nothing completes them, so both waits give up and a
 *               timeout is recorded in the device error word (read and
 *               cleared by gdn_sync_check).
 *   limit       the poll bound, 1 <= limit <= 1 << 22: the mbarrier wait
 *               gives up after `limit` suspending polls (each suspends for at
 *               most a hardware-defined interval), the counter wait after
 *               4 * limit acquire loads, so the kernel's run time is bounded.
 *   waits_ok    host pointer to 2 ints or NULL: whether the mbarrier wait and
 *               the counter wait succeeded (1) or gave up (0).
 *   stream      cudaStream_t to enqueue on; the call synchronises it.
 * Returns GDN_OK once the kernel has finished (a timeout is reported by the
 * following gdn_sync_check, not here), GDN_ERR_INVALID_ARG for a limit or
 * `complete` out of range, GDN_ERR_CUDA if the launch or the copy failed.
 */
gdn_status gdn_selftest_wait(int complete, long long limit, int *waits_ok, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_SELFTEST_H */
