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

#ifdef __cplusplus
}
#endif

#endif /* KDA_TESTING_H */
