/*
 * sdv_testing.h -- test hooks of libsdv.so (declared apart from sdv.h: they
 * exist so that tests can reach paths a correct call never takes).
 *
 * Every device wait in the library (on an mbarrier, a node weight written by
 * another CTA, or a request's node count) gives up after a limit, marks the
 * requests it served SDV_DEV_TIMEOUT in *device_status and lets the kernel
 * return, so that a wait which never ends cannot hang the GPU.  These hooks
 * make such a wait run out on purpose, without any fault: the waited-for
 * flag is simply never set.
 */
#ifndef SDV_TESTING_H
#define SDV_TESTING_H

#include "sdv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Limit, in nanoseconds, of every bounded device wait in later calls made
 * from the calling host thread; 0 restores the default of 2 s.  Returns
 * SDV_OK. */
int sdv_testing_set_wait_limit(unsigned long long wait_ns);

/* The LM-head kernels (sdv_verify_greedy_lm_head, sdv_lm_head_logits,
 * sdv_lm_head_trie_logits) run as CTA pairs (tcgen05 cta_group::2, 256-row
 * tiles over two SMs) wherever a cluster of two CTAs fits, and as one CTA
 * per 128-row tile otherwise.  on = 1 makes every later launch in the
 * process take the one-CTA form, so that tests cover it on a device where
 * pairs fit; on = 0 restores the default.  Not thread-safe against
 * concurrent launches.  Returns SDV_OK. */
int sdv_testing_set_lm_head_single_cta(int on);

/* sdv_verify_block or sdv_verify_multidraft (mode SDV_MODE_BLOCK or
 * SDV_MODE_MULTIDRAFT; arguments as there) with the trie roots taken out of
 * the node kernel's work list.  Every node below a root then waits for a
 * weight its parent never writes, and every request's decision waits for
 * node records that never come: all those waits run out at the limit, the
 * call ends with SDV_DEV_TIMEOUT in *device_status, and each request whose
 * length is at least 1 comes back invalid (accept_len 0, accept_draft 0,
 * out_token -1, accept_prob and residual_mass 0).  The workspace is left in
 * no state a later call depends on.  Returns as the sdv_verify_* calls;
 * SDV_ERR_INVALID also for any other mode. */
int sdv_testing_verify_without_roots(int mode, SDV_VERIFY_ARGS);

#ifdef __cplusplus
}
#endif
#endif
