// Prefill: chunked (WY / UT) form of the KDA recurrence on tcgen05 tensor
// cores.  One persistent CTA per (sequence, head) walks its chunks of C = 64
// tokens in order; the fp32 state lives in tensor memory (TMEM) for the whole
// sequence and meets HBM only at the start and the end.
//
// Per chunk, with k^, q^ the normalised conv outputs, v the conv output of v,
// g the per-channel log-decay, G_r = sum_{i<=r} g_i (inclusive, per channel)
// and S0 the state entering the chunk ("Kimi K3 Metal Gap Analysis", section
// 2 "KDA Attention", row "Recurrence", unrolled over the chunk):
//
//   A'[r,i] = sum_c k^_r[c] k^_i[c] e^{G_r[c]-G_i[c]}   (i <  r)
//   P [r,i] = sum_c q^_r[c] k^_i[c] e^{G_r[c]-G_i[c]}   (i <= r)
//   Minv    = (I + Diag(beta) A')^{-1}                    (unit lower triangular)
//   U       = Minv Diag(beta) (V - K_g S0),  K_g[r] = k^_r e^{G_r}
//   O_pre   = Q_g S0 + P U,                  Q_g[r] = q^_r e^{G_r}
//   S_new   = Diag(e^{G_last}) S0 + K_dec^T U,  K_dec[r] = k^_r e^{G_last - G_r}
//
// The decay factors are split around a per-channel reference rho:
//   L = [k^ e^{G-rho}; q^ e^{G-rho}] (128 x 128),  R = k^ e^{rho-G} (64 x 128)
// so that [A'; P] = L R^T is ONE dense MMA, L (Diag(e^rho) S0) gives
// [K_g S0; Q_g S0] in ONE MMA, and K_dec = e^{G_last-rho} R.  With rho =
// G_last / 2 every factor lies in [e^{-80}, e^{80}] as long as the chunk's
// total decay per channel is at most 160 (always true for ordinary inputs);
// a chunk beyond that computes A' and P exactly (pairwise exponentials on
// CUDA cores) and uses rho_L = 0, rho_R = G_last, where every factor is <= 1.
//
// MMAs per chunk (all kind::tf32, fp32 accumulate, M = 128):
//   MMA0  D0 = L R^T                                  (N = 64,  K = 128)
//   MMA_T DT = [I; P] Minv          A from TMEM       (N = 64,  K = 64)
//   MMA1  D1 = L (Diag(e^rho) S0)                     (N = 128, K = 128)
//   MMA2  D1 += DT (Diag(beta) X)   A from TMEM       (N = 128, K = 64)
//         with D1's top half cleared after X = V - K_g S0 was read, so D1 =
//         [U; O_pre]
//   MMA3  M  += R^T U               A from TMEM       (N = 128, K = 64)
//         on the TMEM master M = Diag(e^rho) S0; then S_new = e^{G_last-rho} M.
// The unit-lower inverse is a forward substitution on CUDA cores.
#include "kda_internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int D = kHeadDim;  // 128
constexpr int C = kChunk;    // 64
constexpr int kThreads = 256;
constexpr float kMaxSpan = 160.0f;

// Dynamic shared memory map (bytes).
constexpr uint32_t OFF_ST = 0;                // (Diag(e^rho) S0)^T operand, N=128 x K=128 tf32
constexpr uint32_t OFF_L = OFF_ST + 65536;    // L operand 128 x 128; staging of y_k / y_q
constexpr uint32_t OFF_R = OFF_L + 65536;     // R operand 64 x 128; staging of G; then
                                              // Diag(beta) A' (fp32 64x64); then the
                                              // Diag(beta) X / U operand N=128 x K=64
constexpr uint32_t OFF_V = OFF_R + 32768;     // v conv output, fp32 64 x 128 (SW128 layout)
constexpr uint32_t OFF_MT = OFF_V + 32768;    // Minv^T operand N=64 x K=64
constexpr uint32_t OFF_SMALL = OFF_MT + 16384;
constexpr uint32_t kSmemBytes = OFF_SMALL + 4096;

// TMEM column map (512 columns allocated).
constexpr int TM_S = 0;     // state master, lane = key channel, column = value channel
constexpr int TM_D1 = 128;  // [K_g S0; Q_g S0] -> [U; O_pre]
constexpr int TM_D0 = 256;  // [A'; P] -> [I; P] (A operand of MMA_T)
constexpr int TM_DT = 320;  // [Minv; P Minv] (A operand of MMA2)
constexpr int TM_RT = 384;  // R^T (A operand of MMA3), lane = channel, column = token

__device__ __forceinline__ float bf16f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) {
    return x > 0.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

template <typename T>
__device__ __forceinline__ T& at(uint8_t* base, uint32_t off) {
    return *reinterpret_cast<T*>(base + off);
}

struct Waiter {
    uint64_t* bar;
    int* dead;  // shared: a bounded wait already gave up in this CTA
    int* err;
    uint32_t phase;
    // Wait for the next MMA commit; bounded, and immediate once the CTA is dead.
    __device__ __forceinline__ void wait() {
        if (!*dead) {
            bool ok = false;
            for (int i = 0; i < (1 << 20); ++i) {
                if (ptx::mbar_try_wait(bar, phase)) { ok = true; break; }
                if ((i & 1023) == 1023 && *(volatile int*)dead) break;
            }
            if (!ok) {
                *(volatile int*)dead = 1;
                atomicOr(err, ptx::kErrPrefillWait);
            }
        }
        phase ^= 1u;
        tc::fence_after();
    }
};

__device__ __forceinline__ void sync_tc() {
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
}

// Operand writes (generic proxy) and TMEM stores made visible to the MMA issuer.
__device__ __forceinline__ void publish() {
    tc::wait_st();
    ptx::fence_proxy_async_smem();
    sync_tc();
}

__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_kernel(const LayerParams p, const PrefillIO io, int* err) {
    extern __shared__ __align__(1024) uint8_t sm[];
    float* s_beta = reinterpret_cast<float*>(sm + OFF_SMALL);   // [64]
    float* s_rq = s_beta + 64;                                    // [64]
    float* s_rk = s_rq + 64;                                      // [64]
    float* s_rhoL = s_rk + 64;                                    // [128]
    float* s_rhoR = s_rhoL + 128;                                 // [128]
    float* s_esc = s_rhoR + 128;                                  // [128] e^{G_last - rho_R}
    float* s_part = s_esc + 128;                                  // [2][64] RMS partial sums
    uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_part + 128);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_bar + 1);
    int* s_dead = reinterpret_cast<int*>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh - b * p.H;
    const int H = p.H, T = io.T;
    const size_t HD = (size_t)H * D, HD3 = 3 * HD;

    if (warp == 0) tc::alloc(s_tmem, 512);
    if (tid == 0) {
        ptx::mbar_init(s_bar, 1);
        ptx::fence_mbar_init();
        *s_dead = 0;
    }
    sync_tc();
    const uint32_t tm = *s_tmem;
    Waiter wt{s_bar, s_dead, err, 0u};

    // Per-thread roles: c = channel for the thread-per-channel passes; the
    // TMEM quadrant of this warp is (warp & 3), its column half is warp >> 2.
    const int c = tid & (D - 1);
    const int half = tid >> 7;
    const int qrow = (warp & 3) * 32 + lane;   // TMEM lane of this thread

    // Initial state into the TMEM master.
    {
        const float* src = io.S + ((size_t)bh * D + qrow) * D + half * 64;
#pragma unroll
        for (int j0 = 0; j0 < 64; j0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v = *reinterpret_cast<const float4*>(src + j0 + j);
                r[j] = __float_as_uint(v.x); r[j + 1] = __float_as_uint(v.y);
                r[j + 2] = __float_as_uint(v.z); r[j + 3] = __float_as_uint(v.w);
            }
            tc::st32(tc::taddr(tm, warp, TM_S + half * 64 + j0), r);
        }
        tc::wait_st();
    }

    // Conv taps, windows and decay constants of this thread's channel(s).
    float* win = io.conv_state + (size_t)b * 3 * HD3;
    float4 w_a, w_b;            // half 0: taps of q and k; half 1: taps of v
    float wa[3], wb[3];         // windows (oldest first)
    float expA = 0.f, dtb = 0.f;
    {
        const size_t ga = (size_t)(half == 0 ? 0 : 2) * HD + (size_t)h * D + c;
        const size_t gb = HD + (size_t)h * D + c;   // k (half 0 only)
        w_a = *reinterpret_cast<const float4*>(p.conv_w + ga * 4);
        w_b = *reinterpret_cast<const float4*>(p.conv_w + gb * 4);
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            wa[j] = win[j * HD3 + ga];
            wb[j] = win[j * HD3 + gb];
        }
        if (half == 1) {
            expA = expf(p.A_log[h * D + c]);
            dtb = p.dt_bias[h * D + c];
        }
    }

    const int nchunks = (T + C - 1) / C;
    for (int ci = 0; ci < nchunks; ++ci) {
        const int t0 = ci * C;
        const int n = min(C, T - t0);
        const size_t row0 = ((size_t)(b * T + t0) * H + h) * D;   // token t0, channel 0
        const size_t tstride = HD;                                   // elements between tokens

        // ---- A1: conv + SiLU per channel over the chunk; decay and its cumulative sum.
        bool big = false;
        if (half == 0) {
            float xq[C], xk[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                xq[r] = r < n ? bf16f(io.q[row0 + r * tstride + c]) : 0.f;
                xk[r] = r < n ? bf16f(io.k[row0 + r * tstride + c]) : 0.f;
            }
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float yq = 0.f, yk = 0.f;
                if (r < n) {
                    const float pq = fmaf(w_a.w, xq[r], fmaf(w_a.z, wa[2], fmaf(w_a.y, wa[1], w_a.x * wa[0])));
                    const float pk = fmaf(w_b.w, xk[r], fmaf(w_b.z, wb[2], fmaf(w_b.y, wb[1], w_b.x * wb[0])));
                    yq = siluf_(pq);
                    yk = siluf_(pk);
                    wa[0] = wa[1]; wa[1] = wa[2]; wa[2] = xq[r];
                    wb[0] = wb[1]; wb[1] = wb[2]; wb[2] = xk[r];
                }
                at<float>(sm, OFF_L + tc::sw128(r, c, 128)) = yk;
                at<float>(sm, OFF_L + tc::sw128(C + r, c, 128)) = yq;
            }
        } else {
            float xv[C], xz[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                xv[r] = r < n ? bf16f(io.v[row0 + r * tstride + c]) : 0.f;
                xz[r] = r < n ? io.z[row0 + r * tstride + c] : 0.f;
            }
            float G = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float yv = 0.f;
                if (r < n) {
                    const float pv = fmaf(w_a.w, xv[r], fmaf(w_a.z, wa[2], fmaf(w_a.y, wa[1], w_a.x * wa[0])));
                    yv = siluf_(pv);
                    wa[0] = wa[1]; wa[1] = wa[2]; wa[2] = xv[r];
                    G += -expA * softplusf_(xz[r] + dtb);
                }
                at<float>(sm, OFF_V + tc::sw128(r, c, C)) = yv;
                at<float>(sm, OFF_R + tc::sw128(r, c, C)) = G;
            }
            big = -G > kMaxSpan;
            s_esc[c] = G;   // G_last for now
        }
        const bool fb = __syncthreads_or(big) != 0;
        if (half == 1) {
            const float G = s_esc[c];
            const float rl = fb ? 0.f : 0.5f * G;
            const float rr = fb ? G : 0.5f * G;
            s_rhoL[c] = rl;
            s_rhoR[c] = rr;
            s_esc[c] = expf(G - rr);
        }

        // ---- A2: per-token norms of the conv outputs and beta.
        if (tid < 2 * C) {
            const int r = tid & (C - 1);
            const int rowL = tid < C ? r : C + r;   // y_k rows first, then y_q
            float ss = 0.f;
#pragma unroll
            for (int k4 = 0; k4 < D; k4 += 4) {
                const float4 v = at<float4>(sm, OFF_L + tc::sw128(rowL, k4, 128));
                ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
            }
            (tid < C ? s_rk : s_rq)[r] = 1.0f / sqrtf(ss + p.l2_eps);
        } else if (tid < 3 * C) {
            const int r = tid - 2 * C;
            s_beta[r] = r < n ? sigmoidf_(io.beta_logit[((size_t)(b * T + t0 + r)) * H + h]) : 0.f;
        }
        __syncthreads();

        // ---- A2b (rare): exact [A'; P] when the chunk decays by more than kMaxSpan.
        if (fb) {
            const int R = tid & 127;           // D0 row: A' rows 0..63, P rows 64..127
            const int r = R & (C - 1);
            const bool isP = R >= C;
            const float rn = isP ? s_rq[r] : s_rk[r];
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
            for (int ch = 0; ch < D; ++ch) {
                const float a = at<float>(sm, OFF_L + tc::sw128(R, ch, 128));
                const float gr = at<float>(sm, OFF_R + tc::sw128(r, ch, C));
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int col = half * 32 + i;
                    if (isP ? col <= r : col < r) {
                        const float kk = at<float>(sm, OFF_L + tc::sw128(col, ch, 128));
                        const float gi = at<float>(sm, OFF_R + tc::sw128(col, ch, C));
                        acc[i] = fmaf(a * kk, expf(gr - gi), acc[i]);
                    }
                }
            }
            uint32_t out[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) out[i] = __float_as_uint(acc[i] * rn * s_rk[half * 32 + i]);
            tc::st32(tc::taddr(tm, warp, TM_D0 + half * 32), out);
            tc::wait_st();
            __syncthreads();
        }

        // ---- A3: L, R (shared memory, in place over the staging) and R^T (TMEM).
        {
            const float rl = s_rhoL[c], rr = s_rhoR[c];
            uint32_t rt[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int r = half * 32 + i;
                const uint32_t oK = OFF_L + tc::sw128(r, c, 128);
                const uint32_t oQ = OFF_L + tc::sw128(C + r, c, 128);
                const uint32_t oR = OFF_R + tc::sw128(r, c, C);
                const float G = at<float>(sm, oR);
                const float kh = at<float>(sm, oK) * s_rk[r];
                const float qh = at<float>(sm, oQ) * s_rq[r];
                const float eL = expf(G - rl);
                const float eR = expf(rr - G);
                at<uint32_t>(sm, oK) = tc::f2tf32(kh * eL);
                at<uint32_t>(sm, oQ) = tc::f2tf32(qh * eL);
                const uint32_t rv = tc::f2tf32(kh * eR);
                at<uint32_t>(sm, oR) = rv;
                rt[i] = rv;
            }
            tc::st32(tc::taddr(tm, warp, TM_RT + half * 32), rt);
        }
        publish();

        // ---- MMA0: [A'; P] = L R^T.
        if (!fb) {
            if (tid == 0) {
                constexpr uint32_t id = tc::idesc_tf32(128, 64);
#pragma unroll
                for (int ks = 0; ks < D / 8; ++ks) {
                    const int kb = ks >> 2, kin = ks & 3;
                    tc::mma_ss(tm + TM_D0,
                               tc::desc_sw128(ptx::smem_u32(sm + OFF_L + kb * 16384 + kin * 32)),
                               tc::desc_sw128(ptx::smem_u32(sm + OFF_R + kb * 8192 + kin * 32)), id,
                               ks > 0);
                }
                tc::commit(s_bar);
            }
            wt.wait();
        }

        // ---- C1: Diag(beta) A' to shared memory, D0 -> [I; P] in TMEM.
        if (warp < 4) {
            float* sM = reinterpret_cast<float*>(sm + OFF_R);   // [64][64], R is no longer needed
            if (warp < 2) {
                const int r = qrow;   // 0..63
                const float br = s_beta[r];
#pragma unroll
                for (int i0 = 0; i0 < C; i0 += 32) {
                    uint32_t v[32];
                    tc::ld32(tc::taddr(tm, warp, TM_D0 + i0), v);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int col = i0 + i;
                        sM[r * C + col] = col < r ? br * __uint_as_float(v[i]) : 0.f;
                        v[i] = col == r ? tc::f2tf32(1.0f) : 0u;
                    }
                    tc::st32(tc::taddr(tm, warp, TM_D0 + i0), v);
                }
            } else {
                const int r = qrow - C;   // P row
#pragma unroll
                for (int i0 = 0; i0 < C; i0 += 32) {
                    uint32_t v[32];
                    tc::ld32(tc::taddr(tm, warp, TM_D0 + i0), v);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = (i0 + i) <= r ? tc::f2tf32(__uint_as_float(v[i])) : 0u;
                    tc::st32(tc::taddr(tm, warp, TM_D0 + i0), v);
                }
            }
        }
        tc::wait_st();
        sync_tc();

        // ---- C2: Minv = (I + Diag(beta) A')^{-1}, one column per thread
        //      (forward substitution), written as the N=64 x K=64 operand Minv^T.
        if (tid < C) {
            const float* sM = reinterpret_cast<const float*>(sm + OFF_R);
            const int j = tid;
            float x[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float s = r == j ? 1.0f : 0.0f;
#pragma unroll
                for (int i = 0; i < r; ++i) s = fmaf(-sM[r * C + i], x[i], s);
                x[r] = s;
            }
#pragma unroll
            for (int i = 0; i < C; i += 4) {
                uint4 u;
                u.x = tc::f2tf32(x[i]); u.y = tc::f2tf32(x[i + 1]);
                u.z = tc::f2tf32(x[i + 2]); u.w = tc::f2tf32(x[i + 3]);
                at<uint4>(sm, OFF_MT + tc::sw128(j, i, C)) = u;
            }
        }
        publish();

        // ---- MMA_T: [Minv; P Minv] = [I; P] Minv.
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 64);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ts(tm + TM_DT, tm + TM_D0 + ks * 8,
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_MT + kb * 8192 + kin * 32)), id, ks > 0);
            }
            tc::commit(s_bar);
        }
        wt.wait();

        // ---- C4 + D: round DT to tf32 in place; state pass: S^T operand
        //      scaled by e^{rho_L}, master scaled by e^{rho_R}.
        {
            uint32_t v[32];
            tc::ld32(tc::taddr(tm, warp, TM_DT + half * 32), v);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = tc::f2tf32(__uint_as_float(v[i]));
            tc::st32(tc::taddr(tm, warp, TM_DT + half * 32), v);

            const float eL = expf(s_rhoL[qrow]);
            const float eR = expf(s_rhoR[qrow]);
#pragma unroll
            for (int j0 = 0; j0 < 64; j0 += 32) {
                uint32_t s[32];
                tc::ld32(tc::taddr(tm, warp, TM_S + half * 64 + j0), s);
                tc::wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 64 + j0 + jj;
                    const float sv = __uint_as_float(s[jj]);
                    at<uint32_t>(sm, OFF_ST + tc::sw128(j, qrow, 128)) = tc::f2tf32(sv * eL);
                    s[jj] = __float_as_uint(sv * eR);
                }
                tc::st32(tc::taddr(tm, warp, TM_S + half * 64 + j0), s);
            }
        }
        publish();

        // ---- MMA1: D1 = L (Diag(e^rho_L) S0) = [K_g S0; Q_g S0].
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 128);
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ss(tm + TM_D1,
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_L + kb * 16384 + kin * 32)),
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_ST + kb * 16384 + kin * 32)), id, ks > 0);
            }
            tc::commit(s_bar);
        }
        wt.wait();

        // ---- E: X = V - K_g S0 -> Diag(beta) X operand (N=128 x K=64); clear D1 top.
        if ((warp & 3) < 2) {
            const int r = qrow;   // token
            const float br = s_beta[r];
#pragma unroll
            for (int j0 = 0; j0 < 64; j0 += 32) {
                uint32_t v[32];
                tc::ld32(tc::taddr(tm, warp, TM_D1 + half * 64 + j0), v);
                tc::wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; jj += 4) {
                    const int j = half * 64 + j0 + jj;
                    const float4 vv = at<float4>(sm, OFF_V + tc::sw128(r, j, C));
                    at<uint32_t>(sm, OFF_R + tc::sw128(j, r, 128)) =
                        tc::f2tf32(br * (vv.x - __uint_as_float(v[jj])));
                    at<uint32_t>(sm, OFF_R + tc::sw128(j + 1, r, 128)) =
                        tc::f2tf32(br * (vv.y - __uint_as_float(v[jj + 1])));
                    at<uint32_t>(sm, OFF_R + tc::sw128(j + 2, r, 128)) =
                        tc::f2tf32(br * (vv.z - __uint_as_float(v[jj + 2])));
                    at<uint32_t>(sm, OFF_R + tc::sw128(j + 3, r, 128)) =
                        tc::f2tf32(br * (vv.w - __uint_as_float(v[jj + 3])));
                }
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) v[jj] = 0u;
                tc::st32(tc::taddr(tm, warp, TM_D1 + half * 64 + j0), v);
            }
        }
        publish();

        // ---- MMA2: D1 += [Minv; P Minv] Diag(beta) X = [U; P U].
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 128);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ts(tm + TM_D1, tm + TM_DT + ks * 8,
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_R + kb * 16384 + kin * 32)), id, 1u);
            }
            tc::commit(s_bar);
        }
        wt.wait();

        // ---- F: U -> operand of MMA3; O_pre -> RMSNorm, gamma, gate -> o.
        float op[64];
        if ((warp & 3) < 2) {
            const int r = qrow;
#pragma unroll
            for (int j0 = 0; j0 < 64; j0 += 32) {
                uint32_t v[32];
                tc::ld32(tc::taddr(tm, warp, TM_D1 + half * 64 + j0), v);
                tc::wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    at<uint32_t>(sm, OFF_R + tc::sw128(half * 64 + j0 + jj, r, 128)) =
                        tc::f2tf32(__uint_as_float(v[jj]));
            }
        } else {
            const int r = qrow - C;
            float ss = 0.f;
#pragma unroll
            for (int j0 = 0; j0 < 64; j0 += 32) {
                uint32_t v[32];
                tc::ld32(tc::taddr(tm, warp, TM_D1 + half * 64 + j0), v);
                tc::wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    op[j0 + jj] = __uint_as_float(v[jj]);
                    ss = fmaf(op[j0 + jj], op[j0 + jj], ss);
                }
            }
            s_part[half * C + r] = ss;
        }
        publish();   // U operand visible; partial sums visible

        // ---- MMA3 (issued now, overlaps the output epilogue): M += R^T U.
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 128);
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ts(tm + TM_S, tm + TM_RT + ks * 8,
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_R + kb * 16384 + kin * 32)), id, 1u);
            }
            tc::commit(s_bar);
        }
        if ((warp & 3) >= 2) {
            const int r = qrow - C;
            if (r < n) {
                const float ms = (s_part[r] + s_part[C + r]) * (1.0f / D);
                const float inv = 1.0f / sqrtf(ms + p.rms_eps);
                const size_t orow = row0 + (size_t)r * tstride + half * 64;
                const float* gl = io.gate_logit + orow;
                const float* gm = p.gamma + h * D + half * 64;
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const float4 g = *reinterpret_cast<const float4*>(gl + j);
                    const float4 gg = *reinterpret_cast<const float4*>(gm + j);
                    float4 o;
                    o.x = gg.x * op[j] * inv * sigmoidf_(g.x);
                    o.y = gg.y * op[j + 1] * inv * sigmoidf_(g.y);
                    o.z = gg.z * op[j + 2] * inv * sigmoidf_(g.z);
                    o.w = gg.w * op[j + 3] * inv * sigmoidf_(g.w);
                    *reinterpret_cast<float4*>(io.o + orow + j) = o;
                }
            }
        }
        wt.wait();

        // ---- G: S_new = e^{G_last - rho_R} M.
        {
            const float e = s_esc[qrow];
#pragma unroll
            for (int j0 = 0; j0 < 64; j0 += 32) {
                uint32_t s[32];
                tc::ld32(tc::taddr(tm, warp, TM_S + half * 64 + j0), s);
                tc::wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) s[jj] = __float_as_uint(__uint_as_float(s[jj]) * e);
                tc::st32(tc::taddr(tm, warp, TM_S + half * 64 + j0), s);
            }
        }
        tc::wait_st();
        sync_tc();
    }

    // Final state and conv window back to global memory.
    {
        float* dst = io.S + ((size_t)bh * D + qrow) * D + half * 64;
#pragma unroll
        for (int j0 = 0; j0 < 64; j0 += 32) {
            uint32_t s[32];
            tc::ld32(tc::taddr(tm, warp, TM_S + half * 64 + j0), s);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(dst + j0 + j) =
                    make_float4(__uint_as_float(s[j]), __uint_as_float(s[j + 1]),
                                __uint_as_float(s[j + 2]), __uint_as_float(s[j + 3]));
        }
        const size_t ga = (size_t)(half == 0 ? 0 : 2) * HD + (size_t)h * D + c;
        const size_t gb = HD + (size_t)h * D + c;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            win[j * HD3 + ga] = wa[j];
            if (half == 0) win[j * HD3 + gb] = wb[j];
        }
    }
    sync_tc();
    if (warp == 0) tc::dealloc(tm, 512);
}

bool g_attr_done[64] = {};

}  // namespace

size_t prefill_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_prefill(const LayerParams& p, const PrefillIO& io, const DeviceInfo& dev,
                           int* err_word, cudaStream_t stream) {
    const long long grid = (long long)io.B * p.H;
    if (grid <= 0 || io.T <= 0) return cudaSuccess;
    if (dev.device < 0 || dev.device >= 64 || !g_attr_done[dev.device]) {
        cudaError_t e = cudaFuncSetAttribute(kda_prefill_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev.device >= 0 && dev.device < 64) g_attr_done[dev.device] = true;
    }
    kda_prefill_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(p, io, err_word);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
