/*
 * moe_testing.h — test hooks of the MoE layer library (not for production).
 */
#ifndef MOE_GB300_TESTING_H
#define MOE_GB300_TESTING_H

#ifdef __cplusplus
extern "C" {
#endif

/* Make moe_stage_experts() fail with MOE_ERR_STAGING once n copies have been
 * queued in one call (n = 0: the first copy fails; n < 0: hook off).  Lets a
 * test exercise the staging error path on the host, with no GPU fault. */
void moe_testing_fail_copies_after(int n);

#ifdef __cplusplus
}
#endif

#endif
