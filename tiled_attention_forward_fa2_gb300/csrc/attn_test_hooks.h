/*
 * attn_test_hooks.h -- extra entry point of the TEST build of the library
 * (lib/libattn_fwd_gb300_testhooks.so, compiled with -DATTN_TEST_HOOKS).  The
 * production library neither declares nor contains it.
 *
 * attn_test_withhold_kv -- nonzero: every later forward launch issues no K/V
 * tile loads, so its pipeline waits can never complete and run into their
 * bound (lower it with attn_set_tuning); the kernel then records
 * ATTN_ERR_TIMEOUT for attn_last_status, drains what it has in flight, frees
 * its tensor memory and returns.  Zero restores normal launches.  This is how
 * the timeout path is exercised on a GPU without faulting it.
 */
#ifndef ATTN_FWD_GB300_TEST_HOOKS_H
#define ATTN_FWD_GB300_TEST_HOOKS_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

attn_status_t attn_test_withhold_kv(int on);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_GB300_TEST_HOOKS_H */
