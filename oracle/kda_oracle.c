/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY (see kda_oracle.h).
 *
 * The KDA token step written out literally, one (sequence, head) at a time,
 * one token at a time, in double precision.  No chunking, no fusion, no
 * reordering: every quantity is formed the way the defining table states it.
 * Independent (sequence, head) pairs may run on separate threads; nothing is
 * shared between them but read-only parameters.
 *
 * Readings of the sources, where they are silent or garbled:
 *  - Decay: the gap analysis prints a garbled decay formula (a stray factor
 *    and no softplus); the sign-safe form gk = -exp(A_log) * softplus(z +
 *    dt_bias) is used, with z the low-rank decay input (W_fb W_fa x).
 *  - beta = sigmoid(beta_logit) scales both the erase and the write term of
 *    the recurrence.  The recurrence row omits it; the token-0 check in
 *    "Correctness" divides the output by v*beta, which needs it.
 *  - Read-out uses the state after the update (again fixed by that check).
 *  - State orientation: S is [key channel][value channel]; o = S^T q and the
 *    decay scales rows (the "St*q" of the "O projection" row).
 *  - No 1/sqrt(d) scale on q (the token-0 identity holds only without one).
 *  - L2 normalisation: x / sqrt(sum x^2 + l2_eps).
 *  - RMSNorm over the d value channels of one head, gamma per (head, channel).
 *  - Conv: depthwise, width 4, causal, no bias, SiLU after it, applied to q,
 *    k and v; the window keeps the previous 3 pre-conv inputs, oldest first.
 */
#include "kda_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef __linux__
#include <sched.h>
#endif

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double silu(double x) { return x * sigmoid(x); }

/* ln(1 + e^x), evaluated without overflow for large |x|. */
static double softplus(double x)
{
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/*
 * bfloat16: 1 sign bit, the 8 exponent bits of IEEE binary32 and 7 stored
 * fraction bits, i.e. binary32 with 8 significant bits.  Normal values are
 * m * 2^(E-7) with m in [128, 255] and E in [-126, 127]; subnormals are
 * m * 2^-133 with m in [0, 127].  Rounding is to nearest, ties to the even
 * m; a magnitude that rounds to 2^128 or above becomes infinity.  The bit
 * pattern is the upper half of the binary32 pattern of the same value.
 */
uint16_t kda_oracle_bf16_round(double x)
{
    if (isnan(x)) return 0x7FC0;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    const double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);                   /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    if (E < -126) E = -126;         /* the subnormal spacing is that of E = -126 */
    const double spacing = ldexp(1.0, E - 7);
    const double m = a / spacing;   /* exact: a power-of-two scaling */
    const double r = nearbyint(m);  /* to nearest, ties to even (default mode) */
    const double val = r * spacing;
    if (val >= ldexp(1.0, 128)) return sign | 0x7F80;
    const float f = (float)val;     /* exact: every bfloat16 value is a binary32 value */
    uint32_t bits;
    memcpy(&bits, &f, sizeof(bits));
    return (uint16_t)(sign | (bits >> 16));
}

double kda_oracle_bf16_value(uint16_t b)
{
    const uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof(f));
    return (double)f;
}

void kda_oracle_bf16_round_n(size_t n, const double *x, uint16_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = kda_oracle_bf16_round(x[i]);
}

void kda_oracle_bf16_value_n(size_t n, const uint16_t *b, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = kda_oracle_bf16_value(b[i]);
}

typedef struct {
    int B, T, H, d;
    const double *q, *k, *v, *z, *beta_logit, *gate_logit;
    const double *conv_w, *dt_bias, *A_log, *gamma;
    double l2_eps, rms_eps;
    double *conv_state, *S, *o, *o_pre;
    double *qhat, *khat, *vconv, *gk_out, *beta_out;
    int state_bf16;   /* store S as bfloat16 between tokens */
} job_t;

/*
 * "Conv4 + SiLU" row: causal depthwise convolution of width 4 over the token
 * axis, per channel, followed by SiLU.  `tensor` selects q (0), k (1) or v (2).
 * Reads the window of the previous three inputs and shifts the new input in.
 */
static void conv4_silu(const job_t *J, int b, int h, int tensor,
                       const double *x_t, double *y)
{
    const int H = J->H, d = J->d;
    const size_t HD3 = (size_t)3 * H * d;
    double *win = J->conv_state + (size_t)b * 3 * HD3;
    for (int c = 0; c < d; ++c) {
        const size_t ch = (size_t)tensor * H * d + (size_t)h * d + c;
        const double *w = J->conv_w + ch * 4;
        double x_m3 = win[0 * HD3 + ch];
        double x_m2 = win[1 * HD3 + ch];
        double x_m1 = win[2 * HD3 + ch];
        double pre = w[0] * x_m3 + w[1] * x_m2 + w[2] * x_m1 + w[3] * x_t[c];
        y[c] = silu(pre);
        win[0 * HD3 + ch] = x_m2;
        win[1 * HD3 + ch] = x_m1;
        win[2 * HD3 + ch] = x_t[c];
    }
}

/* "L2 normalize q/k" row: per-head L2 normalisation over the d channels. */
static void l2_normalize(double *x, int d, double eps)
{
    double ss = 0.0;
    for (int c = 0; c < d; ++c) ss += x[c] * x[c];
    double inv = 1.0 / sqrt(ss + eps);
    for (int c = 0; c < d; ++c) x[c] *= inv;
}

/* One (sequence b, head h) over all T tokens. */
static void run_head(const job_t *J, int b, int h)
{
    const int T = J->T, H = J->H, d = J->d;
    double *qv = malloc(sizeof(double) * d);
    double *kv = malloc(sizeof(double) * d);
    double *vv = malloc(sizeof(double) * d);
    double *a = malloc(sizeof(double) * d);
    double *gkv = malloc(sizeof(double) * d);
    double *u = malloc(sizeof(double) * d);
    double *op = malloc(sizeof(double) * d);
    double *S = J->S + ((size_t)b * H + h) * (size_t)d * d;

    for (int t = 0; t < T; ++t) {
        const size_t row = (((size_t)b * T + t) * H + h) * (size_t)d;
        const size_t bth = ((size_t)b * T + t) * H + h;

        /* Conv4 + SiLU on q, k and v. */
        conv4_silu(J, b, h, 0, J->q + row, qv);
        conv4_silu(J, b, h, 1, J->k + row, kv);
        conv4_silu(J, b, h, 2, J->v + row, vv);

        /* L2 normalise q and k (v is left as it is). */
        l2_normalize(qv, d, J->l2_eps);
        l2_normalize(kv, d, J->l2_eps);

        /* "Decay compute": per-channel log-decay gk and decay a = e^gk. */
        for (int c = 0; c < d; ++c) {
            gkv[c] = -exp(J->A_log[(size_t)h * d + c]) *
                     softplus(J->z[row + c] + J->dt_bias[(size_t)h * d + c]);
            a[c] = exp(gkv[c]);
        }
        const double beta = sigmoid(J->beta_logit[bth]);

        /*
         * "Recurrence": S <- (I - beta k k^T) Diag(e^gk) S + beta k v^T.
         * First S' = Diag(a) S (rows are key channels).  Then
         * (I - beta k k^T) S' = S' - beta k (k^T S'), with u = k^T S'.
         */
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) S[(size_t)i * d + j] *= a[i];
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += kv[i] * S[(size_t)i * d + j];
            u[j] = s;
        }
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j)
                S[(size_t)i * d + j] += -beta * kv[i] * u[j] + beta * kv[i] * vv[j];

        /* "O projection" without the W_o / W_g matmuls: o_pre = S^T q. */
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += S[(size_t)i * d + j] * qv[i];
            op[j] = s;
        }
        /* Head RMSNorm with gamma, then the sigmoid output gate. */
        double ms = 0.0;
        for (int j = 0; j < d; ++j) ms += op[j] * op[j];
        ms /= d;
        const double inv_rms = 1.0 / sqrt(ms + J->rms_eps);
        for (int j = 0; j < d; ++j) {
            J->o[row + j] = J->gamma[(size_t)h * d + j] * op[j] * inv_rms *
                            sigmoid(J->gate_logit[row + j]);
            if (J->o_pre) J->o_pre[row + j] = op[j];
        }

        /* bfloat16 state: the token's arithmetic and read-out use the new
         * state as computed; what is kept for the next token is its
         * rounding to bfloat16. */
        if (J->state_bf16)
            for (size_t i = 0; i < (size_t)d * d; ++i)
                S[i] = kda_oracle_bf16_value(kda_oracle_bf16_round(S[i]));

        if (J->qhat) memcpy(J->qhat + row, qv, sizeof(double) * d);
        if (J->khat) memcpy(J->khat + row, kv, sizeof(double) * d);
        if (J->vconv) memcpy(J->vconv + row, vv, sizeof(double) * d);
        if (J->gk_out) memcpy(J->gk_out + row, gkv, sizeof(double) * d);
        if (J->beta_out) J->beta_out[bth] = beta;
    }
    free(qv); free(kv); free(vv); free(a); free(gkv); free(u); free(op);
}

typedef struct {
    const job_t *J;
    int first, step;
} worker_t;

static void *worker(void *arg)
{
    const worker_t *w = arg;
    const int n = w->J->B * w->J->H;
    for (int p = w->first; p < n; p += w->step) run_head(w->J, p / w->J->H, p % w->J->H);
    return NULL;
}

/*
 * Low-rank front-end ("What runs where (per layer)", row "KDA low-rank
 * (fa,fb,bp)"; "Decay compute" row: z = W_fb W_fa x).  Each product is a
 * plain sum over its inner index, one token at a time.
 */
int kda_oracle_lowrank(int N, int hidden, int rank, int H, int d,
                       const double *x, const double *W_fa, const double *W_fb,
                       const double *W_bp, double *z, double *beta_logit)
{
    if (N < 0 || hidden <= 0 || rank <= 0 || H <= 0 || d <= 0) return -1;
    if (N == 0) return 0;
    if (!x || !W_fa || !W_fb || !W_bp || !z || !beta_logit) return -1;
    const size_t HD = (size_t)H * d;
    double *u = malloc(sizeof(double) * rank);
    for (int n = 0; n < N; ++n) {
        const double *xn = x + (size_t)n * hidden;
        for (int r = 0; r < rank; ++r) {
            double s = 0.0;
            for (int j = 0; j < hidden; ++j) s += W_fa[(size_t)r * hidden + j] * xn[j];
            u[r] = s;
        }
        for (size_t m = 0; m < HD; ++m) {
            double s = 0.0;
            for (int r = 0; r < rank; ++r) s += W_fb[m * rank + r] * u[r];
            z[(size_t)n * HD + m] = s;
        }
        for (int h = 0; h < H; ++h) {
            double s = 0.0;
            for (int j = 0; j < hidden; ++j) s += W_bp[(size_t)h * hidden + j] * xn[j];
            beta_logit[(size_t)n * H + h] = s;
        }
    }
    free(u);
    return 0;
}

/*
 * Projections ("What runs where (per layer)", row "KDA projections
 * (q,k,v,g,o)"; "O projection" row): y = W x, one token at a time, each
 * output a plain sum over the input index.
 */
int kda_oracle_project(int N, int in, int out, const double *x, const double *W, double *y)
{
    if (N < 0 || in <= 0 || out <= 0) return -1;
    if (N == 0) return 0;
    if (!x || !W || !y) return -1;
    for (int n = 0; n < N; ++n) {
        const double *xn = x + (size_t)n * in;
        for (int i = 0; i < out; ++i) {
            const double *wi = W + (size_t)i * in;
            double s = 0.0;
            for (int j = 0; j < in; ++j) s += wi[j] * xn[j];
            y[(size_t)n * out + i] = s;
        }
    }
    return 0;
}

int kda_oracle_cpu_count(void)
{
#ifdef __linux__
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) return CPU_COUNT(&set);
#endif
    return 1;
}

static int run_all(int B, int T, int H, int d,
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
                   int nthreads, int state_bf16)
{
    if (B < 0 || T < 0 || H <= 0 || d <= 0) return -1;
    if (B == 0 || T == 0) return 0;
    if (!q || !k || !v || !z || !beta_logit || !gate_logit || !conv_w ||
        !dt_bias || !A_log || !gamma || !conv_state || !S || !o)
        return -1;
    job_t J = {B, T, H, d, q, k, v, z, beta_logit, gate_logit, conv_w,
               dt_bias, A_log, gamma, l2_eps, rms_eps, conv_state, S, o,
               o_pre, qhat, khat, vconv, gk, beta, state_bf16};
    const int n = B * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = n;
    if (nthreads == 1) {
        worker_t w = {&J, 0, 1};
        worker(&w);
        return 0;
    }
    pthread_t *tid = malloc(sizeof(pthread_t) * nthreads);
    worker_t *ws = malloc(sizeof(worker_t) * nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        ws[i].J = &J;
        ws[i].first = i;
        ws[i].step = nthreads;
        if (pthread_create(&tid[i], NULL, worker, &ws[i]) != 0) break;
        ++started;
    }
    /* Any slot that could not get a thread is run here. */
    for (int i = started; i < nthreads; ++i) worker(&ws[i]);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    free(ws);
    return 0;
}

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
                   int nthreads)
{
    return run_all(B, T, H, d, q, k, v, z, beta_logit, gate_logit, conv_w, dt_bias, A_log, gamma,
                   l2_eps, rms_eps, conv_state, S, o, o_pre, qhat, khat, vconv, gk, beta,
                   nthreads, 0);
}

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
                              int nthreads)
{
    return run_all(B, T, H, d, q, k, v, z, beta_logit, gate_logit, conv_w, dt_bias, A_log, gamma,
                   l2_eps, rms_eps, conv_state, S, o, o_pre, qhat, khat, vconv, gk, beta,
                   nthreads, 1);
}
