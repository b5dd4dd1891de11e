/*
 * kda_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, sequential, double-precision CPU definition of the Kimi Delta
 * Attention (KDA) token step.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path never
 * does.  It shares no code, header or constant with the CUDA library.
 *
 * Sources (page title, then section/table/row):
 *   "Kimi K3 Metal Gap Analysis", section 2 "KDA Attention (kda_forward)",
 *     rows "Conv4 + SiLU", "L2 normalize q/k", "Decay compute",
 *     "Recurrence", "O projection".
 *   "Metal (Apple GPU) backend for Kimi K3", table "What runs where (per
 *     layer)" (low-rank fa/fb/bp feed the decay and beta) and section
 *     "Correctness" (token-0 zero-state identity, which fixes beta and the
 *     read-out-after-update order).
 *
 * All arrays are dense, row-major, double, host memory, owned by the caller.
 * Shapes (B sequences, T tokens, H heads, d = head dimension):
 *   q, k, v, z, gate_logit : [B][T][H][d]      (pre-conv q/k/v)
 *   beta_logit             : [B][T][H]
 *   conv_w                 : [3][H*d][4]       (q, k, v; tap 3 = current token)
 *   dt_bias, A_log, gamma  : [H][d]
 *   conv_state             : [B][3][3*H*d]     (oldest tap first; in/out)
 *   S                      : [B][H][d][d]      (row = key channel, col = value channel; in/out)
 *   o, o_pre               : [B][T][H][d]      (o_pre may be NULL)
 *   qhat, khat, vconv, gk  : [B][T][H][d]      (optional intermediates, may be NULL)
 *   beta                   : [B][T][H]         (optional, may be NULL)
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Returns 0 on success, -1 on a bad argument. */
int kda_oracle_run(int B, int T, int H, int d,
                   const double *q, const double *k, const double *v,
                   const double *z, const double *beta_logit,
                   const double *gate_logit,
                   const double *conv_w, const double *dt_bias,
                   const double *A_log, const double *gamma,
                   double l2_eps, double rms_eps,
                   double *conv_state, double *S,
                   double *o, double *o_pre,
                   double *qhat, double *khat, double *vconv,
                   double *gk, double *beta,
                   int nthreads);

/*
 * Low-rank front-end of the decay and beta inputs ("Metal (Apple GPU) backend
 * for Kimi K3", table "What runs where (per layer)", row "KDA low-rank
 * (fa,fb,bp)"; "Kimi K3 Metal Gap Analysis", section 2, row "Decay compute",
 * whose z is W_fb W_fa x).  For each of N tokens with hidden input x:
 *   u          = W_fa x           u: [rank]
 *   z          = W_fb u           z: [H*d]   (head h, channel c at h*d + c)
 *   beta_logit = W_bp x           beta_logit: [H]
 * Shapes: x [N][hidden], W_fa [rank][hidden], W_fb [H*d][rank],
 * W_bp [H][hidden]; z [N][H*d] and beta_logit [N][H] are written.
 * Returns 0 on success, -1 on a bad argument.
 */
int kda_oracle_lowrank(int N, int hidden, int rank, int H, int d,
                       const double *x, const double *W_fa, const double *W_fb,
                       const double *W_bp, double *z, double *beta_logit);

/*
 * Projections on either side of the token step ("Metal (Apple GPU) backend
 * for Kimi K3", table "What runs where (per layer)", row "KDA projections
 * (q,k,v,g,o)"; "Kimi K3 Metal Gap Analysis", section 2, row "O projection":
 * W_o[sig(W_g x) * RMSNorm_head(S^T q)]).  A plain product y = W x per token:
 *   x [N][in], W [out][in], y [N][out]:  y[n][i] = sum_j W[i][j] x[n][j].
 * The input projections are this with W the rows of W_q, W_k, W_v and W_g;
 * the output projection is this with W = W_o and x the gated, normalised o.
 * Returns 0 on success, -1 on a bad argument.
 */
int kda_oracle_project(int N, int in, int out, const double *x, const double *W, double *y);

/*
 * The same T tokens with the state stored as bfloat16 between tokens: each
 * token runs in double precision from the stored state, its read-out uses
 * the new state as computed, and the new state is then rounded to bfloat16
 * (to nearest, ties to even) for the next token.  S comes in as bfloat16
 * values (doubles that kda_oracle_bf16_round maps to themselves) and goes out
 * rounded.  This is the storage of the "Zero-copy state persistence" and
 * "Wrap-once buffer cache" notes of "Metal (Apple GPU) backend for Kimi K3"
 * (model-lifetime state kept across tokens) at half the bytes; the pages
 * give no state precision, so the rounding point is this reading.
 * Returns 0 on success, -1 on a bad argument.
 */
int kda_oracle_run_bf16_state(int B, int T, int H, int d,
                              const double *q, const double *k, const double *v,
                              const double *z, const double *beta_logit,
                              const double *gate_logit,
                              const double *conv_w, const double *dt_bias,
                              const double *A_log, const double *gamma,
                              double l2_eps, double rms_eps,
                              double *conv_state, double *S,
                              double *o, double *o_pre,
                              double *qhat, double *khat, double *vconv,
                              double *gk, double *beta,
                              int nthreads);

/*
 * bfloat16 (binary32's sign and 8 exponent bits, 7 stored fraction bits):
 * kda_oracle_bf16_round rounds a double to nearest, ties to even (overflow
 * to infinity, subnormals kept) and returns the 16-bit pattern;
 * kda_oracle_bf16_value returns the exact value of a pattern.  The _n forms
 * map arrays of n elements.
 */
uint16_t kda_oracle_bf16_round(double x);
double kda_oracle_bf16_value(uint16_t b);
void kda_oracle_bf16_round_n(size_t n, const double *x, uint16_t *out);
void kda_oracle_bf16_value_n(size_t n, const uint16_t *b, double *out);

/* Number of hardware threads this process may run on (sched affinity). */
int kda_oracle_cpu_count(void);

#ifdef __cplusplus
}
#endif
#endif
