/*
 * kda_testing.h -- test hooks exported by libkda.so.  Not part of the public
 * C ABI (include/kda.h); used by the library's own tests only.
 */
#ifndef KDA_TESTING_H
#define KDA_TESTING_H

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launch, on `stream`, one kernel whose bounded wait runs out: it waits at
 * most limit_us microseconds on an mbarrier nothing arrives on (no copy or
 * MMA is pending), sets its bit in the context's error word and returns.  The
 * next kda_sync_status(ctx, stream) returns KDA_ERR_TIMEOUT and clears the
 * word.  limit_us must be in [1, 1000000].
 */
KDA_API kda_status kda_testing_bounded_wait(kda_ctx *ctx, unsigned limit_us, void *stream);

/*
 * Launch policies, computed on the host without a device:
 * kda_testing_prefill_relay_heads: how many of `heads` (sequence, head)
 * pairs of a T-token kda_prefill run on the few-head schedule (the split
 * schedule with a workspace, else relay pairs) on sm_count SMs: all when
 * twice their number fits, else those of a last partial wave that fills at
 * most half of the SMs, none for a single chunk.  kda_testing_project_o_ksplit: the K ranges of kda_project_o on N
 * tokens (2 when its hidden / 128 x token-tile output tiles fill at most half
 * of the SMs and HD spans at least 16 slices of 64, else 1).  -1 on a
 * negative argument.
 */
KDA_API long long kda_testing_prefill_relay_heads(long long heads, int T, int sm_count);
KDA_API int kda_testing_project_o_ksplit(int hidden, int N, int HD, int sm_count);

#ifdef __cplusplus
}
#endif

#endif /* KDA_TESTING_H */
