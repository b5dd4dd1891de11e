/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) token step.
 *
 * What the library computes, per sequence b, head h and token t (d_k = d_v =
 * d = 128), following "Kimi K3 Metal Gap Analysis", section 2 "KDA Attention
 * (kda_forward)":
 *
 *   row "Conv4 + SiLU":      y = SiLU(w0*x[t-3] + w1*x[t-2] + w2*x[t-1] + w3*x[t])
 *                            per channel, for q, k and v (causal, depthwise,
 *                            width 4, no bias; the window keeps the last three
 *                            pre-conv inputs, oldest first)
 *   row "L2 normalize q/k":  q^ = q / sqrt(|q|^2 + l2_eps), same for k
 *   row "Decay compute":     gk = -exp(A_log) * softplus(z + dt_bias) per channel
 *                            (the printed formula is garbled; this is its
 *                            sign-safe form), beta = sigmoid(beta_logit)
 *   row "Recurrence":        S <- (I - beta k^ k^T) Diag(e^gk) S + beta k^ v^T
 *                            (S is d_k x d_v fp32, rows = key channels)
 *   row "O projection":      o = gamma * RMSNorm_head(S^T q^) * sigmoid(gate_logit)
 *                            (the W_o / W_g matmuls stay outside the library;
 *                            the gate logits come in)
 *
 * The read-out uses the updated state and beta scales both the erase and the
 * write term; "Metal (Apple GPU) backend for Kimi K3", section "Correctness"
 * (token-0 zero-state check o / (v * beta) = q^ . k^) fixes both.
 *
 * Conventions shared by every call:
 *  - Pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA tensors), dense
 *    and row-major, 16-byte aligned (beta_logit: 4-byte aligned); a
 *    misaligned pointer gives KDA_ERR_ALIGNMENT and nothing is launched.
 *  - Parameters given to kda_create are BORROWED: they must stay valid and
 *    unchanged until kda_destroy.  State (S) and conv windows are owned by the
 *    caller and updated in place.
 *  - Work is enqueued on the caller's stream (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream) and is asynchronous: the library does
 *    not synchronise and allocates no device memory after kda_create.
 *  - Errors come back as a kda_status; there is no CPU fallback.  Argument
 *    errors are detected on the host before any launch.
 *  - One kda_ctx may be used from one host thread at a time.
 *  - Every wait inside a kernel is bounded (1 s of wall time).  A kernel that
 *    gives up stops issuing copies and tensor-core operations, waits (again
 *    bounded) for the ones it already issued, records the failure in the
 *    context's error word and returns; kda_sync_status then reports
 *    KDA_ERR_TIMEOUT.  What the affected (sequence, head) pairs hold afterwards
 *    is stated per call below.  A wait that gives up means the device did not
 *    complete a copy within a second, so later results on that device deserve
 *    the same suspicion.
 *  - Fault injection for tests: the environment variable KDA_FAULT_INJECT,
 *    read by kda_create, names entry points ("decode", "prefill",
 *    "prefill_varlen", "lowrank", "project", "all"; comma-separated; the
 *    low-rank decode step counts as "decode" and "lowrank") whose launches
 *    that context replaces by cudaErrorLaunchFailure: nothing is launched,
 *    no buffer changes, and the call returns KDA_ERR_CUDA.  The name
 *    "relay_drop" (not part of "all") makes kda_prefill's relay pairs skip
 *    their first state hand-over: the receiving CTA's bounded wait runs out,
 *    both CTAs of the pair give up, and kda_sync_status reports
 *    KDA_ERR_TIMEOUT with the pair's S and window unchanged.  The name
 *    "split_drop" (not part of "all") makes the producers of kda_prefill's
 *    split schedule skip publishing their first chunk: the consumers' bounded
 *    waits run out, with the same report and S and window unchanged.
 *    "split_nofit" (not part of "all") makes kda_prefill treat the split
 *    schedule's launch as not fitting on the device, as when fewer SMs are
 *    available to the process than the device has: the relay pairs run
 *    instead, with the same results.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kda_ctx kda_ctx;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, bad config */
    KDA_ERR_ALIGNMENT = 2,    /* a pointer is not 16-byte (beta_logit: 4-byte) aligned */
    KDA_ERR_UNSUPPORTED = 3,  /* head_dim != 128, chunk_size != 64, no sm_103a device */
    KDA_ERR_CUDA = 4,         /* a CUDA runtime call failed; see kda_last_error_detail() */
    KDA_ERR_TIMEOUT = 5       /* a bounded wait inside a kernel gave up (kda_sync_status) */
} kda_status;

typedef struct {
    int num_heads;   /* H >= 1 */
    int head_dim;    /* d_k = d_v; must be 128 */
    int chunk_size;  /* prefill chunk length; must be 64 */
    float l2_eps;    /* added to |x|^2 in the q/k L2 normalisation (e.g. 1e-6) */
    float rms_eps;   /* added to mean(o^2) in the head RMSNorm (e.g. 1e-6) */
} kda_config;

/*
 * Create a context bound to one layer's parameters (the wrap-once,
 * model-lifetime buffers of "Metal (Apple GPU) backend for Kimi K3", section
 * "Design notes worth a reviewer's eye").  All parameter pointers are device
 * pointers, fp32, borrowed:
 *   conv_w    [3][H*d][4]  depthwise taps for q, k, v; tap 3 multiplies the current token
 *   dt_bias   [H][d]
 *   A_log     [H][d]
 *   rms_gamma [H][d]
 * Allocates a few bytes of device memory for the kernel error word on the
 * current device; the context is tied to that device: a decode or prefill
 * call made while another device is current returns KDA_ERR_INVALID_ARG
 * (kda_last_error_detail names both devices) and launches nothing.
 * Returns KDA_OK and *out, or an error with *out left NULL.
 */
KDA_API kda_status kda_create(const kda_config *cfg, const float *conv_w, const float *dt_bias,
                      const float *A_log, const float *rms_gamma, kda_ctx **out);

/* Release the context (NULL is ignored).  Does not touch borrowed buffers. */
KDA_API void kda_destroy(kda_ctx *ctx);

/* Static, human-readable name of a status. */
KDA_API const char *kda_strerror(kda_status status);

/* Text of the last CUDA error seen by this thread's calls into the library
 * (empty string if none).  Static thread-local storage; do not free. */
KDA_API const char *kda_last_error_detail(void);

/*
 * One decode token for B sequences ("Fused KDA token": conv + SiLU, L2 norm,
 * decay, recurrence, read-out, RMSNorm and gate in ONE kernel launch).
 *   q, k, v      [B][H][d] fp32  pre-conv inputs of this token (in)
 *   z            [B][H][d] fp32  low-rank decay input (in)
 *   beta_logit   [B][H]    fp32  (in)
 *   gate_logit   [B][H][d] fp32  (in)
 *   conv_state   [B][3][3*H*d] fp32  previous three pre-conv inputs of q, k,
 *                            v (channel = tensor*H*d + h*d + c), oldest
 *                            first (in/out)
 *   S            [B][H][d][d] fp32  state, row = key channel (in/out)
 *   o            [B][H][d] fp32  gated, normalised output (out)
 *   o_pre        [B][H][d] fp32  S^T q^ before RMSNorm (out), or NULL
 * B == 0 is a no-op returning KDA_OK.  Outputs must not alias inputs.
 * After a give-up (KDA_ERR_TIMEOUT from kda_sync_status) the affected pairs
 * keep their old S and window and their o / o_pre are not written; the other
 * pairs of the call are computed normally.
 */
KDA_API kda_status kda_decode_step(kda_ctx *ctx, int B,
                           const float *q, const float *k, const float *v,
                           const float *z, const float *beta_logit,
                           const float *gate_logit,
                           float *conv_state, float *S,
                           float *o, float *o_pre, void *stream);

/*
 * kda_decode_step with the state stored as bfloat16: the same token for B
 * sequences, reading S as bf16, running the token in fp32 (the read-out o /
 * o_pre uses the new state as computed) and storing the new state rounded to
 * nearest-even bf16.  Half the state bytes each way, so about half the time
 * of kda_decode_step when the state dominates, and half the memory for the
 * state of every layer kept resident (the model-lifetime state of the
 * "Zero-copy state persistence" and "Wrap-once buffer cache" notes of
 * "Metal (Apple GPU) backend for Kimi K3"; the pages give no state
 * precision, so bf16 storage is this library's variant).  The rounding is
 * an error of up to 2^-9 relative per element per token on top of
 * kda_decode_step's arithmetic.
 *   S            [B][H][d][d] bf16 (raw bit patterns), row = key channel (in/out)
 * Every other argument, the alignment rules, B == 0 and the give-up
 * behaviour are those of kda_decode_step.
 */
KDA_API kda_status kda_decode_step_bf16state(kda_ctx *ctx, int B,
                           const float *q, const float *k, const float *v,
                           const float *z, const float *beta_logit,
                           const float *gate_logit,
                           float *conv_state, uint16_t *S,
                           float *o, float *o_pre, void *stream);

/*
 * Bytes of device workspace with which kda_prefill runs B sequences of T
 * tokens on its split schedule (0 when the call has none: one chunk per
 * sequence, or enough sequence-heads to fill the SMs in whole waves).
 */
KDA_API size_t kda_prefill_workspace_bytes(const kda_ctx *ctx, int B, int T);

/*
 * Prefill: T tokens for each of B sequences at once, chunked (chunk_size
 * tokens per chunk, the WY/UT form of the recurrence above), with the same
 * result as T calls of kda_decode_step up to rounding.
 *   q, k, v      [B][T][H][d] bf16 (raw bit patterns)  pre-conv inputs (in)
 *   z            [B][T][H][d] fp32 (in)
 *   beta_logit   [B][T][H]    fp32 (in)
 *   gate_logit   [B][T][H][d] fp32 (in)
 *   conv_state   [B][3][3*H*d] fp32 (in/out), as for kda_decode_step
 *   S            [B][H][d][d] fp32 (in/out)
 *   o            [B][T][H][d] fp32 (out)
 *   workspace    optional device buffer, 16-byte aligned, of workspace_bytes
 *                bytes (NULL: none); the library's scratch for the call,
 *                ordered on the stream like the call itself.
 * B == 0 or T == 0 is a no-op returning KDA_OK.  Sequence-head pairs fill the
 * SMs one CTA each; those that would leave SMs idle (all of them when two
 * CTAs per pair fit on the device, else those of a last partial wave) run on
 * one of two few-head schedules.  With a workspace of at least
 * kda_prefill_workspace_bytes(ctx, B, T) bytes, producer CTAs build every
 * chunk's state-independent operands in parallel and pass them through the
 * workspace to one consumer CTA per pair, which keeps the state and runs the
 * sequential part (one cooperative launch: all its CTAs are resident at once;
 * it needs the device's SMs free of other work to start); with less, or none,
 * or when that launch cannot be resident at once on the device, two CTAs per
 * pair take alternate chunks and hand the state to each other.
 * All schedules compute the same arithmetic in the same order, so results are
 * bit for bit the same whichever runs.
 * After a give-up (KDA_ERR_TIMEOUT from kda_sync_status) an affected pair
 * stops at the end of a chunk and keeps its old S and window; the o rows of
 * its chunks from the one that gave up onwards hold unspecified values
 * (earlier rows hold their results).
 */
KDA_API kda_status kda_prefill(kda_ctx *ctx, int B, int T,
                       const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const float *z, const float *beta_logit, const float *gate_logit,
                       float *conv_state, float *S, float *o,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Prefill of B packed sequences of different lengths: sequence b is tokens
 * [cu_seqlens[b], cu_seqlens[b+1]) of one token axis of total_T tokens, and
 * the result for it is that of kda_prefill on those tokens alone (the same
 * arithmetic, bit for bit), continuing from its own
 * conv_state[b] and S[b].  This is the recurrence of "Kimi K3 Metal Gap
 * Analysis", section 2 "KDA Attention", row "Recurrence", run per sequence;
 * the packed layout is this library's (the pages process one sequence).
 *   cu_seqlens   [B+1] int32, DEVICE memory, non-decreasing, cu_seqlens[0] = 0
 *                and cu_seqlens[B] = total_T.  Read by the kernel; each
 *                range is clamped to [0, total_T] (a malformed array gives
 *                wrong sequences, never an access outside the arrays).
 *   q, k, v      [total_T][H][d] bf16 (raw bit patterns)  pre-conv inputs (in)
 *   z            [total_T][H][d] fp32 (in)
 *   beta_logit   [total_T][H]    fp32 (in)
 *   gate_logit   [total_T][H][d] fp32 (in)
 *   conv_state   [B][3][3*H*d] fp32 (in/out), as for kda_decode_step
 *   S            [B][H][d][d] fp32 (in/out)
 *   o            [total_T][H][d] fp32 (out)
 * Alignment as for kda_prefill; cu_seqlens 4-byte aligned.  A sequence of
 * length 0 leaves its state and window unchanged; B == 0 or total_T == 0 is a
 * no-op returning KDA_OK.  Needs no workspace.  When twice the number of
 * sequence-heads (B x H) fits on the device's SMs, each runs as two CTAs
 * that take alternate chunks (the relay pairs of kda_prefill); else one CTA
 * each.  Sequences are isolated: no value of one sequence's inputs, not
 * even a NaN or an infinity, changes another sequence's o, S or window.
 * Give-ups behave as for kda_prefill.
 */
KDA_API kda_status kda_prefill_varlen(kda_ctx *ctx, int B, const int32_t *cu_seqlens, int total_T,
                       const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const float *z, const float *beta_logit, const float *gate_logit,
                       float *conv_state, float *S, float *o, void *stream);

/*
 * Bind the low-rank front-end weights of the layer to the context ("Metal
 * (Apple GPU) backend for Kimi K3", table "What runs where (per layer)", row
 * "KDA low-rank (fa,fb,bp)"; "Kimi K3 Metal Gap Analysis", section 2, row
 * "Decay compute", whose decay input is z = W_fb W_fa x).  Per token with
 * hidden input x:  u = W_fa x,  z = W_fb u,  beta_logit = W_bp x.
 *   hidden   width of x; a multiple of 4
 *   rank     inner width of W_fb W_fa; a multiple of 4, at most 512
 *   W_fa     [rank][hidden]  fp32 device pointer, 16-byte aligned, borrowed
 *   W_fb     [H*d][rank]     fp32, row h*d + c feeds head h, channel c
 *   W_bp     [H][hidden]     fp32
 * The pages give neither width; both are the caller's.  Rebinding replaces
 * the previous weights.  Launches nothing.
 */
KDA_API kda_status kda_bind_lowrank(kda_ctx *ctx, int hidden, int rank, const float *W_fa,
                                    const float *W_fb, const float *W_bp);

/* Bytes of device workspace kda_lowrank needs for N tokens (0 if no weights
 * are bound or N <= 0). */
KDA_API size_t kda_lowrank_workspace_bytes(const kda_ctx *ctx, int N);

/*
 * The low-rank front-end for N tokens, on tensor cores (two tf32 GEMMs with
 * fp32 accumulation and a fixed-order reduction):
 *   x            [N][hidden] fp32 (in), 16-byte aligned
 *   z            [N][H][d]   fp32 (out): the decay input of kda_decode_step /
 *                kda_prefill (N = B, or N = B*T with the [B][T][H][d] layout)
 *   beta_logit   [N][H]      fp32 (out), 4-byte aligned
 *   workspace    at least kda_lowrank_workspace_bytes(ctx, N) bytes, 16-byte
 *                aligned, owned by the caller; its contents are scratch
 * N == 0 is a no-op.  KDA_ERR_INVALID_ARG if no weights are bound.
 */
KDA_API kda_status kda_lowrank(kda_ctx *ctx, int N, const float *x, float *z, float *beta_logit,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * Size of the static device array kda_lowrank_noalloc keeps its scratch in
 * (every GPU that loads this library holds it until the process exits).
 */
#define KDA_LOWRANK_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * kda_lowrank without a workspace argument.  The paper has no counterpart:
 * this entry point exists for callers that cannot give the library device
 * memory of its own for a call (a host runtime that passes a plugin only the
 * layer's tensors and owns the rest of the device, or a serving loop that
 * must not allocate once it runs).  Its scratch (the split-K partial sums
 * and u) lives in one file-scope static device array of
 * KDA_LOWRANK_NOALLOC_SCRATCH_BYTES; it calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   x, z, beta_logit   as for kda_lowrank
 * A call whose scratch would exceed the array (it grows with N, rank and H;
 * the K split count is lowered first to make it fit) returns
 * KDA_ERR_INVALID_ARG, launches nothing, and kda_last_error_detail gives the
 * bytes needed and the limit.  The result equals kda_lowrank's within
 * rounding (the K split count may differ, so the order of the partial sums
 * may too).
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with the context's device current); make that
 * first call before any stream capture.  All calls on a device share the
 * array and it keeps the last call's contents: calls that overlap on the GPU
 * (on different streams, or not ordered by one stream) race on it.  N == 0
 * is a no-op.
 */
KDA_API kda_status kda_lowrank_noalloc(kda_ctx *ctx, int N, const float *x, float *z,
                                       float *beta_logit, void *stream);

/* Bytes of device workspace kda_decode_step_lowrank needs for B sequences. */
KDA_API size_t kda_decode_lowrank_workspace_bytes(const kda_ctx *ctx, int B);

/*
 * One decode token whose decay input and beta logits come from the hidden
 * input through the bound low-rank weights: kda_lowrank on the B tokens (z
 * and beta_logit kept in the workspace), then the kda_decode_step kernel on
 * them, both on `stream`.
 *   x            [B][hidden] fp32 (in)
 *   q, k, v, gate_logit, conv_state, S, o, o_pre   as for kda_decode_step
 *   workspace    at least kda_decode_lowrank_workspace_bytes(ctx, B) bytes,
 *                16-byte aligned, owned by the caller
 * B == 0 is a no-op.  Give-ups behave as for kda_decode_step.
 */
KDA_API kda_status kda_decode_step_lowrank(kda_ctx *ctx, int B, const float *x,
                                           const float *q, const float *k, const float *v,
                                           const float *gate_logit, float *conv_state, float *S,
                                           float *o, float *o_pre, void *workspace,
                                           size_t workspace_bytes, void *stream);

/*
 * Bind the layer's projection weights ("Metal (Apple GPU) backend for Kimi
 * K3", table "What runs where (per layer)", row "KDA projections
 * (q,k,v,g,o)"; "Kimi K3 Metal Gap Analysis", section 2, row "O
 * projection": W_o[sig(W_g x) * RMSNorm_head(S^T q)]).  Device pointers,
 * bf16 raw bit patterns, 16-byte aligned, borrowed:
 *   hidden   width of the layer's hidden input x and of y; a multiple of 128
 *   W_qkvg   [4*H*d][hidden]  W_q, W_k, W_v and W_g stacked by rows (row
 *            j*H*d + h*d + c of block j feeds head h, channel c)
 *   W_o      [hidden][H*d]
 * Rebinding replaces the previous weights.  Launches nothing.
 */
KDA_API kda_status kda_bind_projections(kda_ctx *ctx, int hidden, const uint16_t *W_qkvg,
                                        const uint16_t *W_o);

/*
 * Input projections of N tokens on tensor cores (bf16 operands, fp32
 * accumulation): q = W_q x, k = W_k x, v = W_v x, gate_logit = W_g x.
 *   x            [N][hidden] bf16 (in)
 *   q, k, v      [N][H][d]: bf16 when qkv_f32 == 0 (the kda_prefill input
 *                format, rounded to nearest even), fp32 when qkv_f32 != 0
 *                (the kda_decode_step format)
 *   gate_logit   [N][H][d] fp32
 * All 16-byte aligned.  N == 0 is a no-op; KDA_ERR_INVALID_ARG if no
 * weights are bound.
 */
KDA_API kda_status kda_project_qkvg(kda_ctx *ctx, int N, const uint16_t *x, void *q, void *k, void *v,
                                    float *gate_logit, int qkv_f32, void *stream);

/* Bytes of device workspace kda_project_o needs for N tokens (a bf16 copy of o). */
KDA_API size_t kda_project_o_workspace_bytes(const kda_ctx *ctx, int N);

/*
 * Output projection of N tokens: y = W_o o, o rounded to bf16 (nearest even)
 * into the workspace, then bf16 products with fp32 accumulation on tensor
 * cores.
 *   o            [N][H][d] fp32 (in): the o of kda_decode_step / kda_prefill
 *   y            [N][hidden] fp32 (out)
 *   workspace    at least kda_project_o_workspace_bytes(ctx, N) bytes
 * All 16-byte aligned.  N == 0 is a no-op.  When the output tiles would leave
 * most SMs idle (a few tokens), the two halves of W_o's columns run on
 * separate CTAs and are added into y (which the call zeroes first); two
 * addends onto zero give the same sum in either order, so y does not
 * depend on scheduling (sums below 2^-126 in magnitude become zero).
 */
KDA_API kda_status kda_project_o(kda_ctx *ctx, int N, const float *o, float *y, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * Synchronise `stream` and report whether any kernel launched with this
 * context since the last call gave up on a bounded wait (KDA_ERR_TIMEOUT) or
 * raised a CUDA error (KDA_ERR_CUDA).  Clears the error word, so the next
 * call reports only what happened after this one.
 */
KDA_API kda_status kda_sync_status(kda_ctx *ctx, void *stream);

/* Number of kernels this library has launched in this process (all contexts). */
KDA_API uint64_t kda_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
