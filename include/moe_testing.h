/*
 * moe_testing.h — test hooks of the MoE layer library (not for production).
 */
#ifndef MOE_GB300_TESTING_H
#define MOE_GB300_TESTING_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Make moe_stage_experts() fail with MOE_ERR_STAGING once n copies have been
 * queued in one call (n = 0: the first copy fails; n < 0: hook off).  Lets a
 * test exercise the staging error path on the host, with no GPU fault. */
void moe_testing_fail_copies_after(int n);

/* Launch one small kernel that waits on an mbarrier nothing ever arrives on,
 * with the library's bounded wait (about one second of %globaltimer); it then
 * records MOE_ERR_TIMEOUT (detail -3) in the error word of `ws` (a workspace
 * from moe_workspace_size, at least 256 bytes) and returns.  Lets a test check
 * that a device wait that cannot finish ends with a status, never a hang or a
 * trap, and that the context stays usable.  Asynchronous on `stream`; read the
 * status with moe_check.  Returns MOE_ERR_INVALID_ARG for a NULL or unaligned
 * ws, MOE_ERR_CUDA if the launch fails. */
moe_status moe_testing_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/* The tensor-core prefill FFN runs either one CTA per 128-row tile or CTA
 * pairs (clusters of two SMs) on 256-row tiles with the 2-CTA MMA.  mode -1
 * (the default) chooses by the batch; 0 forces single CTAs, 1 pairs (when
 * the device can hold them).  Process-wide; lets a test run both kernels on
 * the same inputs. */
void moe_testing_set_tc_pairs(int mode);

#ifdef __cplusplus
}
#endif

#endif
