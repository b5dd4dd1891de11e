// Prefill: chunked (WY / UT) form of the KDA recurrence on tcgen05 tensor
// cores.  One persistent CTA per (sequence, head) walks its chunks of C = 64
// tokens in order; the fp32 state lives in tensor memory (TMEM) for the whole
// sequence and meets HBM only at the start and the end.  Heads that would
// leave SMs idle run on a few-head schedule instead: producer CTAs build the
// state-independent operands of all chunks in parallel for one consumer CTA
// per head that runs only the state chain (split, with a workspace), or two
// CTAs per head take alternate chunks and hand the state over (relay).  The
// phases below are shared by the three kernels, which therefore compute the
// same arithmetic in the same order.
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
//         on the TMEM master M = Diag(e^rho) S0; S_new = e^{G_last-rho} M, that
//         row scale being applied by the next chunk's pass over the master.
// The unit-lower inverse is a forward substitution on CUDA cores for the
// diagonal 16 x 16 blocks and warp-level tf32 MMAs for the rest.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "kda_internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int D = kHeadDim;  // 128
constexpr int C = kChunk;    // 64
constexpr int kThreads = 512;
constexpr float kMaxSpan = 160.0f;

// Dynamic shared memory map (bytes).
constexpr uint32_t OFF_ST = 0;                // (Diag(e^rho) S0)^T operand, N=128 x K=128 tf32;
                                              // between MMA1 and the state pass it stages the
                                              // next chunk's q, k (bf16) and z (fp32) tiles
constexpr uint32_t OFF_L = OFF_ST + 65536;    // L operand 128 x 128; staging of y_k / y_q
constexpr uint32_t OFF_R = OFF_L + 65536;     // R operand 64 x 128; staging of G; then
                                              // Diag(beta) A' (fp32 64x64); then the
                                              // Diag(beta) X / U operand N=128 x K=64
constexpr uint32_t OFF_V = OFF_R + 32768;     // v conv output, fp32 64 x 128 (SW128 layout)
constexpr uint32_t OFF_MT = OFF_V + 32768;    // Minv^T operand N=64 x K=64; stages the v tile
constexpr uint32_t OFF_SMALL = OFF_MT + 16384;
constexpr uint32_t OFF_WIN = OFF_SMALL + 4096;   // conv window of a chunk's first half, 2 x [3][3][128] fp32
constexpr uint32_t kSmemBytes = OFF_WIN + 2 * 4608;
constexpr uint32_t STG_Q = OFF_ST, STG_K = OFF_ST + 16384, STG_Z = OFF_ST + 32768, STG_V = OFF_MT;
// Gate tile of the chunk, then its output tile: four 64-row x 32-channel SW128
// boxes in the upper half of the L region (free once MMA1 has read it; the
// lower half then holds Diag(beta) X, the B operand of MMA2).
constexpr uint32_t OFF_OG = OFF_L + 32768;
constexpr uint32_t kOGBox = 8192;
constexpr uint32_t kStageBytes = 3 * C * D * 2 + C * D * 4;   // 80 KiB per chunk
constexpr uint32_t kRelayBytes = D * D * 4 + D * 4;             // relay: a state and its row scales

// TMEM column map (512 columns allocated).
constexpr int TM_S = 0;     // state master, lane = key channel, column = value channel
constexpr int TM_D1 = 128;  // [K_g S0; Q_g S0] -> [U; O_pre]
constexpr int TM_D0 = 256;  // [A'; P] -> [I; P] (A operand of MMA_T)
constexpr int TM_DT = 320;  // [Minv; P Minv] (A operand of MMA2)
constexpr int TM_RT = 384;  // R^T (A operand of MMA3), lane = channel, column = token

// Fast-intrinsic forms (relative error ~1e-6, far inside the tf32 operand rounding).
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// Packed pairs of fp32 (fma/mul/add .f32x2) and single-instruction
// approximations of 2^x, log2(x) and tanh(x).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk(float a, float b) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk(f32x2 v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float ex2f_(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2f_(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;   // log2(e)
constexpr float kLn2 = 0.6931471805599453f;     // ln(2)

__device__ __forceinline__ float tanhf_(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// SiLU of a pair given h = x / 2: x sigmoid(x) = h + h tanh(h) (one MUFU op
// per element; measured on GB300, tanh.approx.f32 is within 7.8e-6 of tanh
// over [-20, 20], so SiLU is within 1e-5 absolute).  The conv produces h
// directly from halved taps (exact: a power-of-two scale).
__device__ __forceinline__ f32x2 silu2_of_half(f32x2 hx) {
    float a, b;
    upk(hx, a, b);
    return fma2(hx, pk(tanhf_(a), tanhf_(b)), hx);
}

// softplus of a pair: max(x, 0) + ln(1 + e^{-|x|}).
__device__ __forceinline__ f32x2 softplus2(f32x2 x) {
    float a, b;
    upk(x, a, b);
    const f32x2 ax = pk(fabsf(a), fabsf(b));
    float e0, e1;
    upk(mul2(ax, pk(-kLog2e, -kLog2e)), e0, e1);
    float l0, l1;
    upk(add2(pk(ex2f_(e0), ex2f_(e1)), pk(1.0f, 1.0f)), l0, l1);
    const f32x2 relu = mul2(add2(x, ax), pk(0.5f, 0.5f));
    return fma2(pk(lg2f_(l0), lg2f_(l1)), pk(kLn2, kLn2), relu);
}

// Warp-level D (16 x 8, fp32) += A (16 x 8, tf32, row-major) * B (8 x 8, tf32):
// lane (g = lane / 4, t = lane % 4) holds A (g, t), (g + 8, t), (g, t + 4),
// (g + 8, t + 4); B (t, g), (t + 4, g); D (g, 2t), (g, 2t + 1), (g + 8, 2t),
// (g + 8, 2t + 1).
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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
    // Wait for the next phase of the barrier; gives up after kWaitLimitNs of
    // wall time (then marks the CTA dead so later waits return at once).
    __device__ __forceinline__ void wait() {
        if (!*(volatile int*)dead) {
            if (!ptx::mbar_wait_timed(bar, phase, dead)) {
                *(volatile int*)dead = 1;
                atomicOr(err, ptx::kErrPrefillWait);
            }
        }
        phase ^= 1u;
        tc::fence_after();
    }
};

// Barrier over `count` threads (whole warps) with id `id` (0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrive on named barrier `id` without waiting for it (the threads that
// need the arrivals' earlier shared-memory writes bar.sync on it).
__device__ __forceinline__ void named_barrier_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

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


struct Maps {
    CUtensorMap q, k, v, z;   // 4-D (d, H, T, B) boxes of (128, 1, 64, 1)
    CUtensorMap g, o;         // 4-D (d, H, T, B) boxes of (32, 1, 64, 1), 128-byte swizzle
};

// Issuing threads.  Issuing a group of MMAs stalls the issuing warp for
// about the group's execution time, so MMA1 comes from warp 10 (little work
// in C1 and the inverse's first pass); MMA_T from warp 15 as soon as it has
// written the last inverse block; the staging copies from warp 12 (it waits
// for MMA1 anyway); the output store from warp 3 (an output-epilogue warp);
// MMA0, MMA2 and MMA3 from thread 0 (warp 0 has no rows in the output
// epilogue and skips the gate pass).
constexpr int kIssuerB = 480, kIssuer1 = 320, kStager = 384, kOStore = 96;

// Where the per-CTA scalars and mbarriers live in the small region.
constexpr uint32_t kBarOff = OFF_SMALL + 3328;

// One thread's fixed roles and the CTA's shared-memory pointers.  16 warps:
// warp w reaches TMEM lanes [32 (w % 4), +32) and takes column group w / 4 of
// every TMEM pass; in the thread-per-channel passes the same thread owns
// channel c = its TMEM lane.  In the conv / decay phase, grp 0, 1, 2 run the
// conv of q, k, v and grp 3 the decay, each thread on the channel pair
// (cp, cp + 1) for tokens [32 th, 32 th + 32).
struct Thr {
    uint8_t* sm;
    uint32_t tm;
    int tid, warp, lane;
    int qrow, grp;
    int cp, th, pch;
    uint32_t kpL, kpR;   // swizzled K offsets of the pair in the L (128-row) and R / V (64-row) layouts
    uint32_t kcL, kcR;   // the same for channel c
    int cch;
    float* s_beta;   // [64]
    float* s_rq;     // [64]
    float* s_rk;     // [64]
    float* s_part;   // [4][64] RMS partial sums
    float* s_gh0;    // [128] decay sum over tokens 0..31
    float* s_gh1;    // [128] decay sum over tokens 32..63
    float* s_gam;    // [128] gamma / 2 of this head
    float* s_win;    // [2][3][3][128] conv window of a chunk's first half, by chunk parity
};

__device__ __forceinline__ Thr make_thr(uint8_t* sm) {
    Thr t;
    t.sm = sm;
    t.tm = 0;
    t.tid = (int)threadIdx.x;
    t.warp = t.tid >> 5;
    t.lane = t.tid & 31;
    t.qrow = (t.warp & 3) * 32 + t.lane;
    t.grp = t.warp >> 2;
    t.cp = (t.tid & 63) * 2;
    t.th = (t.tid >> 6) & 1;
    t.pch = (t.cp >> 2) & 7;
    t.kpL = (uint32_t)((t.cp >> 5) * 128 * 128 + (t.cp & 3) * 4);
    t.kpR = (uint32_t)((t.cp >> 5) * 64 * 128 + (t.cp & 3) * 4);
    const int c = t.qrow;
    t.kcL = (uint32_t)((c >> 5) * 128 * 128 + (c & 3) * 4);
    t.kcR = (uint32_t)((c >> 5) * 64 * 128 + (c & 3) * 4);
    t.cch = (c >> 2) & 7;
    t.s_beta = reinterpret_cast<float*>(sm + OFF_SMALL);
    t.s_rq = t.s_beta + 64;
    t.s_rk = t.s_rq + 64;
    t.s_part = t.s_rk + 64;
    t.s_gh0 = t.s_part + 256;
    t.s_gh1 = t.s_gh0 + 128;
    t.s_gam = t.s_gh1 + 128;
    t.s_win = reinterpret_cast<float*>(sm + OFF_WIN);
    return t;
}

__device__ __forceinline__ f32x2 unpk_bf2(uint32_t u) {
    return pk(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// Per-thread constants of the conv / decay phase for head h: the channel
// pair's conv taps (halved: the conv then yields x / 2, the argument SiLU
// takes; tap 3 multiplies the current token) or -exp(A_log) and dt_bias,
// and the pair's offset gcp in a [3][H*d] row of the window.
struct ConvW {
    f32x2 W0, W1, W2, W3, nEA, DTB;
    size_t gcp;
};

__device__ __forceinline__ ConvW conv_consts(const Thr& t, const LayerParams& p, int h, size_t HD) {
    ConvW w;
    w.W0 = w.W1 = w.W2 = w.W3 = 0;
    w.nEA = w.DTB = 0;
    w.gcp = (size_t)(t.grp < 3 ? t.grp : 0) * HD + (size_t)h * D + t.cp;
    if (t.grp < 3) {
        const float4 a = *reinterpret_cast<const float4*>(p.conv_w + w.gcp * 4);
        const float4 bq = *reinterpret_cast<const float4*>(p.conv_w + (w.gcp + 1) * 4);
        w.W0 = pk(0.5f * a.x, 0.5f * bq.x); w.W1 = pk(0.5f * a.y, 0.5f * bq.y);
        w.W2 = pk(0.5f * a.z, 0.5f * bq.z); w.W3 = pk(0.5f * a.w, 0.5f * bq.w);
    } else {
        w.nEA = pk(-expf(p.A_log[h * D + t.cp]), -expf(p.A_log[h * D + t.cp + 1]));
        w.DTB = pk(p.dt_bias[h * D + t.cp], p.dt_bias[h * D + t.cp + 1]);
    }
    return w;
}

// Where the first token half of a chunk finds the three inputs before it:
// this CTA's saved window, the inputs in global memory, or the sequence's
// conv window in global memory (its first chunk).
enum : int { kWinShared = 0, kWinInputs = 1, kWinState = 2 };

// ---- A1: conv + SiLU per channel over the chunk (from the staged tiles)
//      into the L (k, q) and V regions; decay and its cumulative sum into the
//      R region and s_gh0 / s_gh1.  Loads of token group g + 1 are issued
//      before the stores of group g.  xg: this thread's input (q, k or v by
//      grp) at channel cp of the head, rows r3 .. r3 + 2 the three tokens
//      before the chunk (kWinInputs); win: the sequence's conv window
//      (kWinState); wpar: parity of the saved window (kWinShared); save: keep
//      this chunk's last three inputs as the window of parity wpar ^ 1.
//      Returns whether half of the chunk decays by more than kMaxSpan / 2 in
//      one of this thread's channels.
__device__ __forceinline__ bool conv_decay(const Thr& t, const ConvW& w, int n, int wmode, int wpar, bool save,
                                           const uint16_t* xg, size_t r3, size_t HD, const float* win) {
    uint8_t* sm = t.sm;
    const int grp = t.grp, cp = t.cp, th = t.th, pch = t.pch;
    bool big = false;
    if (grp < 3) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(
            sm + (grp == 0 ? STG_Q : (grp == 1 ? STG_K : STG_V))) + (cp >> 1);
        const uint32_t dst = grp == 0 ? OFF_L + t.kpL + C * 128 : (grp == 1 ? OFF_L + t.kpL : OFF_V + t.kpR);
        f32x2 M3, M2, M1;   // window, oldest first
        if (th == 0 && wmode == kWinInputs) {
            M3 = unpk_bf2(*reinterpret_cast<const uint32_t*>(xg + r3 * HD));
            M2 = unpk_bf2(*reinterpret_cast<const uint32_t*>(xg + (r3 + 1) * HD));
            M1 = unpk_bf2(*reinterpret_cast<const uint32_t*>(xg + (r3 + 2) * HD));
        } else if (th == 0 && wmode == kWinState) {
            const size_t HD3 = 3 * HD;
            const float2 a = *reinterpret_cast<const float2*>(win + w.gcp);
            const float2 b = *reinterpret_cast<const float2*>(win + HD3 + w.gcp);
            const float2 c = *reinterpret_cast<const float2*>(win + 2 * HD3 + w.gcp);
            M3 = pk(a.x, a.y); M2 = pk(b.x, b.y); M1 = pk(c.x, c.y);
        } else if (th == 0) {
            const float* ws = t.s_win + (wpar * 9 + grp * 3) * D + cp;
            M3 = pk(ws[0], ws[1]); M2 = pk(ws[D], ws[D + 1]); M1 = pk(ws[2 * D], ws[2 * D + 1]);
        } else {
            M3 = unpk_bf2(src[29 * (D / 2)]); M2 = unpk_bf2(src[30 * (D / 2)]); M1 = unpk_bf2(src[31 * (D / 2)]);
        }
        const int r0 = th * 32;
        uint32_t nxt[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) nxt[i] = src[(r0 + i) * (D / 2)];
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            f32x2 x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = unpk_bf2(nxt[i]);
            if (g < 3) {
#pragma unroll
                for (int i = 0; i < 8; ++i) nxt[i] = src[(r0 + (g + 1) * 8 + i) * (D / 2)];
            }
            f32x2 y[8];
            if (n == C) {   // full chunk: the window shift is register renaming
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    f32x2 pre = mul2(w.W0, M3);
                    pre = fma2(w.W1, M2, pre);
                    pre = fma2(w.W2, M1, pre);
                    pre = fma2(w.W3, x[i], pre);
                    y[i] = silu2_of_half(pre);
                    M3 = M2; M2 = M1; M1 = x[i];
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const bool ok = r0 + g * 8 + i < n;
                    f32x2 pre = mul2(w.W0, M3);
                    pre = fma2(w.W1, M2, pre);
                    pre = fma2(w.W2, M1, pre);
                    pre = fma2(w.W3, x[i], pre);
                    y[i] = ok ? silu2_of_half(pre) : 0ull;
                    if (ok) { M3 = M2; M2 = M1; M1 = x[i]; }
                }
            }
            // row r = r0 + 8 g + i (r & 7 = i): the swizzle only flips address
            // bits 4..6, which the row base leaves clear, so it is one XOR
            const uint32_t rb = dst + (uint32_t)(r0 + g * 8) * 128 + (pch << 4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                at<f32x2>(sm, (rb ^ (uint32_t)(i << 4)) + i * 128) = y[i];
            }
        }
        if (save && th == 1) {   // the next chunk's first half starts from this window
            float* ws = t.s_win + ((wpar ^ 1) * 9 + grp * 3) * D + cp;
            upk(M3, ws[0], ws[1]);
            upk(M2, ws[D], ws[D + 1]);
            upk(M1, ws[2 * D], ws[2 * D + 1]);
        }
    } else {
        const f32x2* src = reinterpret_cast<const f32x2*>(sm + STG_Z) + (cp >> 1);
        const int r0 = th * 32;
        f32x2 G = 0;   // (0, 0)
        f32x2 nxt[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) nxt[i] = src[(r0 + i) * (D / 2)];
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            f32x2 zc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) zc[i] = nxt[i];
            if (g < 3) {
#pragma unroll
                for (int i = 0; i < 8; ++i) nxt[i] = src[(r0 + (g + 1) * 8 + i) * (D / 2)];
            }
            f32x2 gg[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const f32x2 sp = softplus2(add2(zc[i], w.DTB));
                if (r0 + g * 8 + i < n) G = fma2(w.nEA, sp, G);
                gg[i] = G;
            }
            const uint32_t rb = OFF_R + t.kpR + (uint32_t)(r0 + g * 8) * 128 + (pch << 4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                at<f32x2>(sm, (rb ^ (uint32_t)(i << 4)) + i * 128) = gg[i];
            }
        }
        *reinterpret_cast<f32x2*>((th == 0 ? t.s_gh0 : t.s_gh1) + cp) = G;
        float ga, gb;
        upk(G, ga, gb);
        big = -ga > 0.5f * kMaxSpan || -gb > 0.5f * kMaxSpan;   // a half beyond kMaxSpan / 2
    }
    return big;
}

// ---- A2: per-token norms of the conv outputs (4 threads per row, one per
//      32-channel block; the 8 lanes of a quarter warp take 8 rows of one
//      block, so their 16-byte loads hit 8 different bank groups) and beta.
__device__ __forceinline__ void norms(const Thr& t, int n, float blog, float l2_eps) {
    const int tid = t.tid;
    const int R = (tid & 7) + 8 * (tid >> 5), part = (tid >> 3) & 3;   // y_k rows 0..63, y_q rows 64..127
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 v = at<float4>(t.sm, OFF_L + tc::sw128(R, part * 32 + j, 128));
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 8);
    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
    if (part == 0) (R < C ? t.s_rk : t.s_rq)[R & (C - 1)] = rsqrtf(ss + l2_eps);
    if (tid < C) t.s_beta[tid] = tid < n ? sigmoidf_(blog) : 0.f;
}

// ---- D: state pass.  The S^T operand of MMA1 scaled by e^{rho_L} to shared
//      memory and the TMEM master scaled by e^{rho_R} (both also by the
//      previous chunk's pending scale esc_prev).  The state comes from the
//      TMEM master, or (rx: relay launches) from the rows the other CTA
//      stored into the S^T region, which the operand then overwrites.
//      gl: this row's G_last.
__device__ __forceinline__ void state_pass(const Thr& t, float& esc_prev, bool rx, bool fb, float gl,
                                           const float* s_rxesc) {
    uint8_t* sm = t.sm;
    const int qrow = t.qrow;
    uint32_t v[32];
    const int j0 = t.grp * 32;
    const uint32_t ta = tc::taddr(t.tm, t.warp, TM_S + j0);
    if (rx) {
        const uint32_t rb = OFF_ST + (uint32_t)qrow * 512;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
            const uint4 x = at<uint4>(sm, rb + ((uint32_t)(t.grp * 8 + (q4 ^ (qrow & 7))) << 4));
            v[4 * q4] = x.x; v[4 * q4 + 1] = x.y; v[4 * q4 + 2] = x.z; v[4 * q4 + 3] = x.w;
        }
        esc_prev = s_rxesc[qrow];
        __syncthreads();   // every received row is read before the operand overwrites it
    } else {
        tc::ld32(ta, v);
        tc::wait_ld();
    }
    const float eL = esc_prev * (fb ? 1.0f : __expf(0.5f * gl));
    const float eR = esc_prev * __expf(fb ? gl : 0.5f * gl);
    // S^T operand element (row j, K = qrow): K block and chunk are fixed per thread.
    const uint32_t kq = (uint32_t)((qrow >> 5) * 128 * 128 + (qrow & 3) * 4);
    const int kch = (qrow >> 2) & 7;
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int j = j0 + g8 * 8 + i;
            const float sv = __uint_as_float(v[g8 * 8 + i]);
            at<uint32_t>(sm, OFF_ST + kq + j * 128 + ((kch ^ (j & 7)) << 4)) = tc::f2tf32(sv * eL);
            v[g8 * 8 + i] = __float_as_uint(sv * eR);
        }
    }
    tc::st32(ta, v);
}

// ---- A2b (rare): exact [A'; P] when the chunk decays by more than kMaxSpan.
__device__ __forceinline__ void exact_fallback(const Thr& t) {
    uint8_t* sm = t.sm;
    const int R = t.qrow;                // D0 row: A' rows 0..63, P rows 64..127
    const int r = R & (C - 1);
    const bool isP = R >= C;
    const float rn = isP ? t.s_rq[r] : t.s_rk[r];
#pragma unroll 1
    for (int g8 = 0; g8 < 2; ++g8) {
        uint32_t out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int col = t.grp * 16 + g8 * 8 + i;
            float acc = 0.f;
            if (isP ? col <= r : col < r) {
#pragma unroll 4
                for (int ch = 0; ch < D; ++ch) {
                    const float a = at<float>(sm, OFF_L + tc::sw128(R, ch, 128));
                    const float gr = at<float>(sm, OFF_R + tc::sw128(r, ch, C)) + (r >= 32 ? t.s_gh0[ch] : 0.f);
                    const float kk = at<float>(sm, OFF_L + tc::sw128(col, ch, 128));
                    const float gi = at<float>(sm, OFF_R + tc::sw128(col, ch, C)) + (col >= 32 ? t.s_gh0[ch] : 0.f);
                    acc = fmaf(a * kk, expf(gr - gi), acc);
                }
            }
            out[i] = __float_as_uint(acc * rn * t.s_rk[col]);
        }
        tc::st8(tc::taddr(t.tm, t.warp, TM_D0 + t.grp * 16 + g8 * 8), out);
    }
    tc::wait_st();
    __syncthreads();
}

// Layout of a 128-lane x 64-column TMEM operand (DT, R^T) in global memory,
// as the 512 threads hold it: thread (w, l) has lane 32 (w % 4) + l and
// columns 16 (w / 4) + [0, 16), stored as four 16-byte pieces k at float
// ((4 w + k) 32 + l) 4, so that a warp's piece k is 512 contiguous bytes.
__device__ __forceinline__ size_t img_at(const Thr& t, int k) {
    return ((size_t)(t.warp * 4 + k) * 32 + t.lane) * 4;
}

// ---- A3: L, R (shared memory, in place over the staging) and R^T (TMEM, or
//      with RT_GLOBAL the global image rt_img), channel c, tokens
//      [16 grp, 16 grp + 16), 8 at a time.
template <bool RT_GLOBAL>
__device__ __forceinline__ void lr_build(const Thr& t, bool fb, float* rt_img) {
    uint8_t* sm = t.sm;
    const int c = t.qrow, grp = t.grp, cch = t.cch;
    // rho_L = rho_R = G_last / 2, or (0, G_last) on the fallback path
    const float gl = t.s_gh0[c] + t.s_gh1[c];
    const float rl = fb ? 0.f : 0.5f * gl, rr = fb ? gl : 0.5f * gl;
    const float goff = grp >= 2 ? t.s_gh0[c] : 0.f;   // tokens 32..63 add the first half
#pragma unroll 1
    for (int g8 = 0; g8 < 2; ++g8) {
        uint32_t rt[8];
        float g[8], yk[8], yq[8];
        const int r0 = grp * 16 + g8 * 8;
        const float4 nk0 = *reinterpret_cast<const float4*>(t.s_rk + r0), nk1 = *reinterpret_cast<const float4*>(t.s_rk + r0 + 4);
        const float4 nq0 = *reinterpret_cast<const float4*>(t.s_rq + r0), nq1 = *reinterpret_cast<const float4*>(t.s_rq + r0 + 4);
        const float nk[8] = {nk0.x, nk0.y, nk0.z, nk0.w, nk1.x, nk1.y, nk1.z, nk1.w};
        const float nq[8] = {nq0.x, nq0.y, nq0.z, nq0.w, nq1.x, nq1.y, nq1.z, nq1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + i;
            const uint32_t ro = (uint32_t)(r * 128 + ((cch ^ (r & 7)) << 4));
            g[i] = at<float>(sm, OFF_R + t.kcR + ro) + goff;
            yk[i] = at<float>(sm, OFF_L + t.kcL + ro) * nk[i];
            yq[i] = at<float>(sm, OFF_L + t.kcL + C * 128 + ro) * nq[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = grp * 16 + g8 * 8 + i;
            const uint32_t ro = (uint32_t)(r * 128 + ((cch ^ (r & 7)) << 4));
            const float eL = __expf(g[i] - rl);
            const float eR = __expf(rr - g[i]);
            rt[i] = tc::f2tf32(yk[i] * eR);
            at<uint32_t>(sm, OFF_L + t.kcL + ro) = tc::f2tf32(yk[i] * eL);
            at<uint32_t>(sm, OFF_L + t.kcL + C * 128 + ro) = tc::f2tf32(yq[i] * eL);
            at<uint32_t>(sm, OFF_R + t.kcR + ro) = rt[i];
        }
        if constexpr (RT_GLOBAL) {   // columns 8 g8 .. 8 g8 + 7: pieces 2 g8, 2 g8 + 1
            *reinterpret_cast<uint4*>(rt_img + img_at(t, 2 * g8)) = make_uint4(rt[0], rt[1], rt[2], rt[3]);
            *reinterpret_cast<uint4*>(rt_img + img_at(t, 2 * g8 + 1)) = make_uint4(rt[4], rt[5], rt[6], rt[7]);
        } else {
            tc::st8(tc::taddr(t.tm, t.warp, TM_RT + grp * 16 + g8 * 8), rt);
        }
    }
}

// The MMA issue loops below are fully unrolled and add constant offsets to
// one base descriptor per operand: a rolled loop, or a descriptor rebuilt
// from the address per instruction, roughly halves the issue rate.

// ---- MMA0: [A'; P] = L R^T (one thread issues).
__device__ __forceinline__ void mma0(const Thr& t, uint64_t* bar) {
    constexpr uint32_t id = tc::idesc_tf32(128, 64);
    const uint64_t da = tc::desc_sw128(ptx::smem_u32(t.sm + OFF_L));
    const uint64_t db = tc::desc_sw128(ptx::smem_u32(t.sm + OFF_R));
#pragma unroll
    for (int ks = 0; ks < D / 8; ++ks) {
        const int kb = ks >> 2, kin = ks & 3;
        tc::mma_ss(t.tm + TM_D0, tc::desc_add(da, kb * 16384 + kin * 32), tc::desc_add(db, kb * 8192 + kin * 32), id,
                   ks > 0);
    }
    tc::commit(bar);
}

// ---- MMA1: D1 = L (Diag(e^rho_L) S0) = [K_g S0; Q_g S0], K blocks
//      [2 HALF, 2 HALF + 2) (one thread issues; half 1 commits to bar1).
template <int HALF>
__device__ __forceinline__ void mma1_part(const Thr& t, uint64_t* bar1) {
    constexpr uint32_t id = tc::idesc_tf32(128, 128);
    const uint64_t da = tc::desc_sw128(ptx::smem_u32(t.sm + OFF_L));
    const uint64_t db = tc::desc_sw128(ptx::smem_u32(t.sm + OFF_ST));
#pragma unroll
    for (int ks = HALF * 8; ks < HALF * 8 + 8; ++ks) {
        const int kb = ks >> 2, kin = ks & 3;
        tc::mma_ss(t.tm + TM_D1, tc::desc_add(da, kb * 16384 + kin * 32), tc::desc_add(db, kb * 16384 + kin * 32), id,
                   ks > 0);
    }
    if (HALF == 1) tc::commit(bar1);
}

// ---- C1: N = Diag(beta) A' to shared memory as N^T (row b holds column b
//      of N; 64-row SW128 layout), D0 -> [I; P] in TMEM (row qrow, columns
//      [16 grp, 16 grp + 16)).
__device__ __forceinline__ void c1_pass(const Thr& t) {
    uint8_t* sm = t.sm;
    const int qrow = t.qrow;
    const bool isA = qrow < C;
    const int r = isA ? qrow : qrow - C;
    const float br = t.s_beta[r];
    const int i0 = t.grp * 16;
    uint32_t v[16];
    tc::ld16(tc::taddr(t.tm, t.warp, TM_D0 + i0), v);
    tc::wait_ld();
    if (isA) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            at<float>(sm, OFF_R + tc::sw128(i0 + i, r, C)) = (i0 + i) < r ? br * __uint_as_float(v[i]) : 0.f;
            v[i] = (i0 + i) == r ? tc::f2tf32(1.0f) : 0u;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = (i0 + i) <= r ? tc::f2tf32(__uint_as_float(v[i])) : 0u;
    }
    tc::st16(tc::taddr(t.tm, t.warp, TM_D0 + i0), v);
}

// ---- C2: Minv = (I + N)^{-1} (N strictly lower) by 16 x 16 blocks.
//      Pass 1: forward substitution with the diagonal block I + N_II on the
//      right-hand sides [I | N_I0 .. N_I(I-1)], giving Minv_II and
//      E_IK = Minv_II N_IK.  Passes 2..4, level by level (I - J = 1, 2, 3):
//      Minv_IJ = -sum_{J <= K < I} E_IK Minv_KJ, one warp per block.  Minv
//      is kept transposed and tf32-rounded in the SW128 layout of the MMA_T
//      operand (row j holds column j of Minv).  Then MMA_T:
//      [Minv; P Minv] = [I; P] Minv, committed to barT.
__device__ __forceinline__ void inverse_mma_t(const Thr& t, uint64_t* barT) {
    uint8_t* sm = t.sm;
    const int tid = t.tid, warp = t.warp, lane = t.lane;
    auto NT = [&](int row, int k) { return OFF_R + tc::sw128(row, k, C); };    // N^T
    auto MT = [&](int row, int k) { return OFF_MT + tc::sw128(row, k, C); };   // Minv^T
    // E_IK column-major (column stride 24 floats, pair stride 384 floats);
    // (I, K) pairs (1,0) (2,0) (2,1) (3,0) (3,1) (3,2): index I (I - 1) / 2 + K.
    const uint32_t OFF_E = OFF_R + 16384;
    auto EC = [&](int pr, int col, int row) { return OFF_E + (uint32_t)(pr * 384 + col * 24 + row) * 4; };
    if (tid < 160) {
        // block row I takes threads [8 I (I + 1), 8 (I + 1) (I + 2)): column u of [I | N_I*]
        const int I = tid < 16 ? 0 : (tid < 48 ? 1 : (tid < 96 ? 2 : 3));
        const int u = tid - 8 * I * (I + 1);
        const int K = (u >> 4) - 1, cc = u & 15;
        float x[16];
        if (K < 0) {
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) x[rr] = rr == cc ? 1.0f : 0.0f;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = at<float4>(sm, NT(K * 16 + cc, I * 16 + q * 4));   // N[16I + 4q + t][16K + cc]
                x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
            }
        }
#pragma unroll
        for (int i = 0; i < 15; ++i) {
#pragma unroll
            for (int q = (i + 1) >> 2; q < 4; ++q) {
                const float4 v = at<float4>(sm, NT(I * 16 + i, I * 16 + q * 4));   // N[16I + 4q + t][16I + i]
                const float nv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int tt = 0; tt < 4; ++tt)
                    if (4 * q + tt > i) x[4 * q + tt] = fmaf(-nv[tt], x[i], x[4 * q + tt]);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {   // tf32-rounded: operands of the level MMAs and of MMA_T
            const uint4 u4 = make_uint4(tc::f2tf32(x[4 * q]), tc::f2tf32(x[4 * q + 1]),
                                        tc::f2tf32(x[4 * q + 2]), tc::f2tf32(x[4 * q + 3]));
            at<uint4>(sm, K < 0 ? MT(I * 16 + cc, I * 16 + q * 4) : EC((I * (I - 1)) / 2 + K, cc, q * 4)) = u4;
        }
    } else {
        // zero the blocks above the diagonal of Minv (K block < row block of Minv^T)
        for (int it = tid - 160; it < 384; it += kThreads - 160) {
            const int pr = it >> 6, rr = (it >> 2) & 15, q = it & 3;
            const int J = pr < 1 ? 1 : (pr < 3 ? 2 : 3);
            const int I = pr - (J * (J - 1)) / 2;
            at<float4>(sm, MT(J * 16 + rr, I * 16 + q * 4)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    ptx::fence_proxy_async_smem();   // Minv^T blocks: smem operand of MMA_T
    __syncthreads();
    // Levels, on warps 15, 14, 11 (blocks J = 0, 1, 2), which have no rows in
    // the X epilogue running meanwhile: warp J computes the 16 x 16 block
    // Minv_{J+lev, J} with warp-level m16n8k8 tf32 MMAs (operands stored
    // tf32-rounded; the result is rounded once more when stored).
    const int J = warp == 15 ? 0 : (warp == 14 ? 1 : (warp == 11 ? 2 : -1));
    if (J >= 0) {
#pragma unroll
        for (int lev = 1; lev < 4; ++lev) {
            if (J < 4 - lev) {
                const int I = J + lev, g = lane >> 2, t4 = lane & 3;
                float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int kk = 0; kk < lev; ++kk) {
                    const int K = J + kk, pr = (I * (I - 1)) / 2 + K;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const int m0 = ks * 8;
                        // A = E_IK rows (g, g + 8), columns (m0 + t4, m0 + t4 + 4)
                        const uint32_t a[4] = {at<uint32_t>(sm, EC(pr, m0 + t4, g)),
                                               at<uint32_t>(sm, EC(pr, m0 + t4, g + 8)),
                                               at<uint32_t>(sm, EC(pr, m0 + t4 + 4, g)),
                                               at<uint32_t>(sm, EC(pr, m0 + t4 + 4, g + 8))};
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)   // B = Minv_KJ rows (m0 + t4, + 4), column 8 nt + g
                            mma_tf32_16x8x8(d[nt], a, at<uint32_t>(sm, MT(J * 16 + nt * 8 + g, K * 16 + m0 + t4)),
                                            at<uint32_t>(sm, MT(J * 16 + nt * 8 + g, K * 16 + m0 + t4 + 4)));
                    }
                }
                // D rows (g, g + 8), columns (8 nt + 2 t4, + 1) -> Minv^T rows 16 J + column
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int cA = J * 16 + nt * 8 + 2 * t4;
                    at<uint32_t>(sm, MT(cA, I * 16 + g)) = tc::f2tf32(-d[nt][0]);
                    at<uint32_t>(sm, MT(cA + 1, I * 16 + g)) = tc::f2tf32(-d[nt][1]);
                    at<uint32_t>(sm, MT(cA, I * 16 + g + 8)) = tc::f2tf32(-d[nt][2]);
                    at<uint32_t>(sm, MT(cA + 1, I * 16 + g + 8)) = tc::f2tf32(-d[nt][3]);
                }
            }
            ptx::fence_proxy_async_smem();   // Minv^T is the smem operand of MMA_T
            if (lev < 3) named_barrier_sync(1, 96);
        }
        // ---- MMA_T: [Minv; P Minv] = [I; P] Minv, issued by the warp that
        //      wrote the last block (runs under the rest of the X epilogue).
        if (tid == kIssuerB) {
            tc::fence_after();
            constexpr uint32_t id = tc::idesc_tf32(128, 64);
            const uint64_t db = tc::desc_sw128(ptx::smem_u32(sm + OFF_MT));
#pragma unroll
            for (int ks = 0; ks < C / 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ts(t.tm + TM_DT, t.tm + TM_D0 + ks * 8, tc::desc_add(db, kb * 8192 + kin * 32), id, ks > 0);
            }
            tc::commit(barT);
        }
    }
}

// DT -> tf32 (A operand of MMA2): in place, or (GLOBAL) into the global image dt_img.
template <bool GLOBAL>
__device__ __forceinline__ void dt_to_tf32(const Thr& t, float* dt_img) {
    uint32_t v[16];
    const uint32_t ta = tc::taddr(t.tm, t.warp, TM_DT + t.grp * 16);
    tc::ld16(ta, v);
    tc::wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = tc::f2tf32(__uint_as_float(v[i]));
    if constexpr (GLOBAL) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(dt_img + img_at(t, k)) = make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    } else {
        tc::st16(ta, v);
    }
}

// ---- E (lane quadrants 0, 1): X = V - K_g S0 -> Diag(beta) X, the B
//      operand of MMA2 (N = 128 value channels x 2 K blocks of 32 tokens,
//      16 KiB each) at x_off; clear D1 top.
__device__ __forceinline__ void x_epilogue(const Thr& t, const float* beta, uint32_t x_off) {
    uint8_t* sm = t.sm;
    const int r = t.qrow;   // token
    const int grp = t.grp;
    const float br = beta[r];
    const uint32_t kr = x_off + (uint32_t)((r >> 5) * 16384 + grp * 32 * 128 + (r & 3) * 4);
    const int rch = (r >> 2) & 7;
    const uint32_t vrow = OFF_V + r * 128;
    uint32_t v[32];
    const uint32_t ta = tc::taddr(t.tm, t.warp, TM_D1 + grp * 32);
    tc::ld32(ta, v);
    const uint32_t vb = vrow + grp * 64 * 128;   // V columns grp * 32 .. + 32 (one K block)
    tc::wait_ld();
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
        const float4 v0 = at<float4>(sm, vb + (((2 * g8) ^ (r & 7)) << 4));
        const float4 v1 = at<float4>(sm, vb + (((2 * g8 + 1) ^ (r & 7)) << 4));
        const float xs[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {   // row j = grp * 32 + 8 g8 + i of the operand (j & 7 = i)
            at<uint32_t>(sm, kr + (g8 * 8 + i) * 128 + ((rch ^ i) << 4)) =
                tc::f2tf32(br * (xs[i] - __uint_as_float(v[g8 * 8 + i])));
            v[g8 * 8 + i] = 0u;
        }
    }
    tc::st32(ta, v);
}

// ---- MMA2: D1 += [Minv; P Minv] Diag(beta) X = [U; P U] (N = 128: a tf32
//      MMA costs about the same per instruction at N = 64 and 128).
__device__ __forceinline__ void mma2(const Thr& t, uint32_t x_off, uint64_t* bar2) {
    constexpr uint32_t id = tc::idesc_tf32(128, 128);
    const uint64_t db = tc::desc_sw128(ptx::smem_u32(t.sm + x_off));
#pragma unroll
    for (int ks = 0; ks < C / 8; ++ks) {
        const int kb = ks >> 2, kin = ks & 3;
        tc::mma_ts(t.tm + TM_D1, t.tm + TM_DT + ks * 8, tc::desc_add(db, kb * 16384 + kin * 32), id, 1u);
    }
    tc::commit(bar2);
}

// The gate tile at og_off becomes gamma * sigmoid(gate) in place, rows
// spread over warps 1..15 (warp 0 issues MMA2).
__device__ __forceinline__ void gate_pass(const Thr& t, uint32_t og_off) {
    if (t.warp > 0) {   // lane = (box, 16-byte chunk) of a row: channels 4 lane .. 4 lane + 3
        const int box = t.lane >> 3, ch = t.lane & 7;
        const float4 gm = *reinterpret_cast<const float4*>(t.s_gam + t.lane * 4);
#pragma unroll 1
        for (int r = t.warp - 1; r < C; r += 15) {
            const uint32_t o = og_off + box * kOGBox + r * 128 + ((ch ^ (r & 7)) << 4);
            const float4 gv = at<float4>(t.sm, o);
            at<float4>(t.sm, o) = make_float4(fmaf(gm.x, tanhf_(0.5f * gv.x), gm.x), fmaf(gm.y, tanhf_(0.5f * gv.y), gm.y),
                                              fmaf(gm.z, tanhf_(0.5f * gv.z), gm.z), fmaf(gm.w, tanhf_(0.5f * gv.w), gm.w));
        }
    }
}

// ---- F (lane quadrants 0, 1): U -> MMA3's U operand at u_off, then (thread
//      0, once the 8 warps are done) MMA3: M += R^T U, committed to bar3.
__device__ __forceinline__ void u_operand_mma3(const Thr& t, uint32_t u_off, uint64_t* bar3) {
    uint8_t* sm = t.sm;
    const int r = t.qrow;
    const uint32_t kr = (uint32_t)((r >> 5) * 128 * 128 + (r & 3) * 4);
    const int rch = (r >> 2) & 7;
    uint32_t v[32];
    tc::ld32(tc::taddr(t.tm, t.warp, TM_D1 + t.grp * 32), v);
    tc::wait_ld();
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
        const int j = t.grp * 32 + jj;
        at<uint32_t>(sm, u_off + kr + j * 128 + ((rch ^ (j & 7)) << 4)) = tc::f2tf32(__uint_as_float(v[jj]));
    }
    ptx::fence_proxy_async_smem();
    tc::fence_before();
    named_barrier_sync(2, 256);   // U operand complete
    if (t.tid == 0) {
        tc::fence_after();
        constexpr uint32_t id = tc::idesc_tf32(128, 128);
        const uint64_t db = tc::desc_sw128(ptx::smem_u32(sm + u_off));
#pragma unroll
        for (int ks = 0; ks < C / 8; ++ks) {
            const int kb = ks >> 2, kin = ks & 3;
            tc::mma_ts(t.tm + TM_S, t.tm + TM_RT + ks * 8, tc::desc_add(db, kb * 16384 + kin * 32), id, 1u);
        }
        tc::commit(bar3);
    }
}

// ---- Output epilogue (lane quadrants 2, 3): the O_pre rows' sums of
//      squares, then RMSNorm x gamma sigmoid(gate) -> o, written over the
//      gate tile at og_off and stored by TMA (rows past T clipped by the
//      copy).  direct: the last, partial chunk of a packed sequence stores its
//      rows < n with plain stores (the rows after it belong to the next
//      sequence); orow0: o of token t0 at head h, channel 0.
__device__ __forceinline__ void out_epilogue(const Thr& t, uint32_t og_off, float rms_eps, int n, bool direct,
                                             float* orow0, size_t orow_stride, const Maps& maps, int h, int tok,
                                             int bmap) {
    uint8_t* sm = t.sm;
    const int grp = t.grp;
    const int r = t.qrow - C;
    float ss = 0.f, ss2 = 0.f;
    uint32_t w[32];
    tc::ld32(tc::taddr(t.tm, t.warp, TM_D1 + grp * 32), w);
    tc::wait_ld();
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        ss = fmaf(__uint_as_float(w[i]), __uint_as_float(w[i]), ss);
        ss2 = fmaf(__uint_as_float(w[i + 1]), __uint_as_float(w[i + 1]), ss2);
    }
    t.s_part[grp * C + r] = ss + ss2;
    named_barrier_sync(3, 256);   // the four column groups' partial sums
    const float inv = rsqrtf((t.s_part[r] + t.s_part[C + r] + t.s_part[2 * C + r] + t.s_part[3 * C + r]) *
                                 (1.0f / D) + rms_eps);
    const uint32_t gbase = og_off + grp * kOGBox + r * 128;   // row r of box grp (SW128)
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {
        const uint32_t* v = w + g8 * 8;
        const uint32_t oa_at = gbase + (((2 * g8) ^ (r & 7)) << 4);
        const uint32_t ob_at = gbase + (((2 * g8 + 1) ^ (r & 7)) << 4);
        const float4 ga = at<float4>(sm, oa_at), gb = at<float4>(sm, ob_at);
        const float4 oa = make_float4(ga.x * __uint_as_float(v[0]) * inv, ga.y * __uint_as_float(v[1]) * inv,
                                      ga.z * __uint_as_float(v[2]) * inv, ga.w * __uint_as_float(v[3]) * inv);
        const float4 ob = make_float4(gb.x * __uint_as_float(v[4]) * inv, gb.y * __uint_as_float(v[5]) * inv,
                                      gb.z * __uint_as_float(v[6]) * inv, gb.w * __uint_as_float(v[7]) * inv);
        if (!direct) {
            at<float4>(sm, oa_at) = oa;
            at<float4>(sm, ob_at) = ob;
        } else if (r < n) {
            float* orow = orow0 + (size_t)r * orow_stride + grp * 32 + g8 * 8;
            *reinterpret_cast<float4*>(orow) = oa;
            *reinterpret_cast<float4*>(orow + 4) = ob;
        }
    }
    ptx::fence_proxy_async_smem();
    named_barrier_sync(3, 256);   // the o tile is complete
    if (t.tid == kOStore && !direct) {
#pragma unroll
        for (int j = 0; j < 4; ++j) ptx::tma_store_4d(&maps.o, j * 32, h, tok, bmap, sm + og_off + j * kOGBox);
        ptx::bulk_commit();
    }
}

// Initial state into the TMEM master (row qrow, columns of this group); S
// points at the head's [d][d] state.
__device__ __forceinline__ void state_in(const Thr& t, const float* S) {
    const float* src = S + (size_t)t.qrow * D + t.grp * 32;
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + j);
        r[j] = __float_as_uint(v.x); r[j + 1] = __float_as_uint(v.y);
        r[j + 2] = __float_as_uint(v.z); r[j + 3] = __float_as_uint(v.w);
    }
    tc::st32(tc::taddr(t.tm, t.warp, TM_S + t.grp * 32), r);
    tc::wait_st();
}

// Final state S = esc M (row qrow, columns of this group) and conv window:
// the last three inputs of the sequence (older taps from the initial window
// when T < 3); x: q, k or v by grp at the head, row stride HD.
__device__ __forceinline__ void state_window_out(const Thr& t, float* S, float esc, const uint16_t* x, size_t rowbase,
                                                 int T, size_t HD, float* win, size_t gcp) {
    float* dst = S + (size_t)t.qrow * D + t.grp * 32;
    uint32_t s[32];
    tc::ld32(tc::taddr(t.tm, t.warp, TM_S + t.grp * 32), s);
    tc::wait_ld();
#pragma unroll
    for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(dst + j) =
            make_float4(esc * __uint_as_float(s[j]), esc * __uint_as_float(s[j + 1]),
                        esc * __uint_as_float(s[j + 2]), esc * __uint_as_float(s[j + 3]));
    if (t.grp < 3 && t.th == 0) {
        const size_t HD3 = 3 * HD;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int tt = T - 3 + j;
            float2 w;
            if (tt >= 0) {
                const uint32_t u = *reinterpret_cast<const uint32_t*>(x + (rowbase + tt) * HD + t.cp);
                w = make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
            } else {   // an older tap of the initial window (not yet overwritten: j + T > j)
                w = *reinterpret_cast<const float2*>(win + (j + T) * HD3 + gcp);
            }
            *reinterpret_cast<float2*>(win + j * HD3 + gcp) = w;
        }
    }
}

// RELAY: two CTAs per (sequence, head), one cluster, take alternate chunks
// (CTA role r does the chunks r, r + 2, ...); each builds the
// state-independent part of its chunk (conv, norms, L/R, MMA0, the inverse,
// MMA_T, DT) while the other runs the state chain of the chunk before, then
// takes the state over from it through distributed shared memory, runs the
// chain and hands the state on.
template <bool RELAY>
__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_kernel(const LayerParams p, const PrefillIO io, int* err, const __grid_constant__ Maps maps) {
    extern __shared__ __align__(1024) uint8_t sm[];
    Thr t = make_thr(sm);
    // mbarriers.  Each completes at most one phase per chunk and every thread
    // that waits on one waits on it once per chunk, so no waiter can fall two
    // phases behind (a parity wait would then alias onto a later phase).
    uint64_t* s_bar = reinterpret_cast<uint64_t*>(sm + kBarOff);   // MMA0 done
    uint64_t* s_tbar = s_bar + 1;                                 // input tiles landed
    uint64_t* s_gbar = s_bar + 2;                                 // gate tile landed
    uint64_t* s_tbarT = s_bar + 3;                                // MMA_T done
    uint64_t* s_bar1 = s_bar + 4;                                 // MMA1 done
    uint64_t* s_drain = s_bar + 5;                                // give-up path: MMA issuers drained
    uint64_t* s_bar2 = s_bar + 6;                                 // MMA2 done
    uint64_t* s_bar3 = s_bar + 7;                                 // MMA3 done
    uint64_t* s_rxfull = s_bar + 8;                               // relay: the other CTA's state landed
    uint64_t* s_rxfree = s_bar + 9;                               // relay: the other CTA can take a state
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_bar + 10);
    int* s_dead = reinterpret_cast<int*>(s_tmem + 1);
    int* s_nt = s_dead + 1;                                       // input-tile phases issued
    int* s_ng = s_dead + 2;                                       // gate-tile phases issued
    float* s_rxesc = reinterpret_cast<float*>(s_dead + 3);        // [128] relay: received row scales

    const int tid = t.tid, warp = t.warp;
    const int bh = RELAY ? io.head0 + (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int role = RELAY ? (int)(blockIdx.x & 1) : 0;   // first chunk of this CTA
    constexpr int kStep = RELAY ? 2 : 1;                  // chunks between two of this CTA's
    const int b = bh / p.H, h = bh - b * p.H;
    const int H = p.H;
    // This sequence's tokens: rows [rowbase, rowbase + T) of the token axis.
    // Fixed length: T = io.T, the maps' axes are (d, H, T, B) and the copies
    // address (t, b); packed sequences (cu_seqlens): the maps' axes are
    // (d, H, total, 1), the copies address (tb0 + t, 0), and the range is
    // clamped to [0, total].
    int T = io.T, tb0 = 0, bmap = b;
    size_t rowbase = (size_t)b * io.T;
    if (io.cu_seqlens) {
        const int lo = min(max(io.cu_seqlens[b], 0), io.T);
        const int hi = min(max(io.cu_seqlens[b + 1], lo), io.T);
        T = hi - lo;
        tb0 = lo;
        bmap = 0;
        rowbase = (size_t)lo;
    }
    const size_t HD = (size_t)H * D, HD3 = 3 * HD;
    const int nchunks = (T + C - 1) / C;
    const int qrow = t.qrow, grp = t.grp;

    if (warp == 0) tc::alloc(s_tmem, 512);
    // Staging of chunk ci's input tiles with TMA box loads (rows past T come
    // back as zeros).  q, k, z land in the S^T operand region and may be
    // issued once MMA1 has read it; v lands in the Minv^T region and may be
    // issued once MMA_T has read it.  One barrier phase covers all four.
    // Staged copies and MMAs are issued without looking at *s_dead (a shared
    // load on the issuing thread's path measurably slows every chunk); after
    // a bounded wait gave up, the CTA leaves at the end of that chunk (the
    // vote at the loop's end) and drains what it issued before returning.
    // The counts of issued tile phases let the drain wait for the last ones.
    auto stage_qkz = [&](int ci) {
        if (tid == kStager) {
            ++*s_nt;
            ptx::mbar_arrive_expect_tx(s_tbar, kStageBytes);
            ptx::tma_load_4d(sm + STG_Q, &maps.q, 0, h, tb0 + ci * C, bmap, s_tbar);
            ptx::tma_load_4d(sm + STG_K, &maps.k, 0, h, tb0 + ci * C, bmap, s_tbar);
            ptx::tma_load_4d(sm + STG_Z, &maps.z, 0, h, tb0 + ci * C, bmap, s_tbar);
            ptx::tma_prefetch_4d(&maps.v, 0, h, tb0 + ci * C, bmap);   // v lands later; have it in L2
        }
    };
    auto stage_v = [&](int ci) {   // joins the phase stage_qkz opened for the same chunk
        if (tid == 0) ptx::tma_load_4d(sm + STG_V, &maps.v, 0, h, tb0 + ci * C, bmap, s_tbar);
    };
    if (tid == 0) {
        ptx::mbar_init(s_bar, 1);
        ptx::mbar_init(s_tbar, 1);
        ptx::mbar_init(s_gbar, 1);
        ptx::mbar_init(s_tbarT, 1);
        ptx::mbar_init(s_bar1, 1);
        ptx::mbar_init(s_drain, 3);
        ptx::mbar_init(s_bar2, 1);
        ptx::mbar_init(s_bar3, 1);
        ptx::mbar_init(s_rxfull, 1);
        ptx::mbar_init(s_rxfree, 1);
        ptx::fence_mbar_init();
        *s_dead = 0;
        *s_nt = 0;
        *s_ng = 0;
    }
    if (tid < D) t.s_gam[tid] = 0.5f * p.gamma[h * D + tid];   // gamma sigmoid(g) = s_gam + s_gam tanh(g / 2)
    sync_tc();
    // Relay pairs: the other CTA's barriers are initialised before either
    // CTA touches them (both CTAs of a cluster are scheduled together).
    if constexpr (RELAY) ptx::cluster_sync();
    t.tm = *s_tmem;
    Waiter wt{s_bar, s_dead, err, 0u};
    Waiter wt2{s_bar2, s_dead, err, 0u};
    Waiter wt3{s_bar3, s_dead, err, 0u};
    Waiter wtma{s_tbar, s_dead, err, 0u};
    Waiter wgate{s_gbar, s_dead, err, 0u};
    Waiter wtT{s_tbarT, s_dead, err, 0u};
    Waiter wt1{s_bar1, s_dead, err, 0u};
    Waiter wrx{s_rxfull, s_dead, err, 0u};
    Waiter wfree{s_rxfree, s_dead, err, 0u};
    if (role < nchunks) {
        stage_qkz(role);
        stage_v(role);
    }

    state_in(t, io.S + (size_t)bh * D * D);

    float* win = io.conv_state + (size_t)b * 3 * HD3;
    const ConvW cw = conv_consts(t, p, h, HD);
    if (grp < 3 && t.th == 0) {
#pragma unroll
        for (int j = 0; j < 3; ++j)
            *reinterpret_cast<float2*>(t.s_win + (grp * 3 + j) * D + t.cp) =
                *reinterpret_cast<const float2*>(win + j * HD3 + cw.gcp);
    }
    const uint16_t* xg = (grp == 0 ? io.q : (grp == 1 ? io.k : io.v)) + (size_t)h * D + t.cp;

    float esc_prev = 1.0f;   // pending e^{G_last - rho_R} of the previous chunk, per state row
    // Relay pairs (a cluster of two CTAs): chunk ci's end state goes to the
    // other CTA as the TMEM master M and its pending row scale, so that the
    // next chunk computes exactly what a single CTA would.  M lands in the
    // other CTA's S^T region (free there between its conv phase and its state
    // pass), rows of 512 bytes with the 16-byte chunk index XOR (row & 7);
    // the scales land in s_rxesc.  Each CTA says when its region is free
    // (s_rxfree of the sender) and the stores complete on s_rxfull.
    const uint32_t peer = (uint32_t)(role ^ 1);
    const uint32_t peer_st = RELAY ? ptx::mapa(ptx::smem_u32(sm + OFF_ST), peer) : 0u;
    const uint32_t peer_esc = RELAY ? ptx::mapa(ptx::smem_u32(s_rxesc), peer) : 0u;
    const uint32_t peer_full = RELAY ? ptx::mapa(ptx::smem_u32(s_rxfull), peer) : 0u;
    const uint32_t peer_free = RELAY ? ptx::mapa(ptx::smem_u32(s_rxfree), peer) : 0u;
    int nrx = 0;   // relay: receives this CTA has announced (thread 0)

    for (int ci = role; ci < nchunks; ci += kStep) {
        const int t0 = ci * C;
        const int n = min(C, T - t0);

        // beta logits of the chunk, consumed after the conv phase.
        const float blog = tid < n ? io.beta_logit[(rowbase + t0 + tid) * H + h] : 0.f;
        wtma.wait();
        // The o tile of the chunk before (K blocks 2, 3 of the L region, which
        // the q and k conv write) must have left shared memory.
        if (tid < 256) {
            if (tid == kOStore) ptx::bulk_wait_read_all();
            named_barrier_sync(5, 256);
        }
        // the chunk before ran in the other CTA (relay): its last three inputs from global memory
        const bool big = conv_decay(t, cw, n, (RELAY && ci > 0) ? kWinInputs : kWinShared, ci & 1, true, xg,
                                    rowbase + (size_t)t0 - 3, HD, win);
        // The exact fallback when a chunk's decay may exceed kMaxSpan in some
        // channel (decided per half of the chunk, so conservatively).
        const bool fb = __syncthreads_or(big) != 0;
        // Relay: the staged tiles in the S^T region are consumed, so the other
        // CTA may store the state after chunk ci - 1 there.
        if (RELAY && ci > 0 && tid == 0) {
            ptx::mbar_arrive_expect_tx(s_rxfull, kRelayBytes);
            ptx::mbar_arrive_remote(peer_free);
            ++nrx;
        }

        norms(t, n, blog, p.l2_eps);
        publish();   // norms, beta

        if (fb) exact_fallback(t);
        lr_build<false>(t, fb, nullptr);
        publish();

        // MMA0 is issued by warp 10 (it has little work in C1 and C2) as soon
        // as L and R are complete; every warp then runs the state pass under
        // it (the pass reads and writes only the TMEM master and the S^T
        // region, neither of which MMA0 touches), and warp 10 issues MMA1
        // behind MMA0 (it runs under C1 and the inverse).  The tensor pipe
        // takes MMA0 first, and the issuing thread, held at the pipe's rate,
        // is not one C1 needs.
        if (!fb && tid == (RELAY ? 0 : kIssuer1)) mma0(t, s_bar);
        if constexpr (!RELAY) {
            // ---- D: state pass (relay launches: later, once the state has arrived)
            state_pass(t, esc_prev, false, fb, t.s_gh0[qrow] + t.s_gh1[qrow], s_rxesc);
            publish();   // S^T operand and rescaled master
            if (tid == kIssuer1) {
                mma1_part<0>(t, s_bar1);
                mma1_part<1>(t, s_bar1);
            }
        }
        if (!fb) wt.wait();   // MMA0

        c1_pass(t);
        tc::wait_st();
        sync_tc();

        inverse_mma_t(t, s_tbarT);
        if constexpr (RELAY) {
            // MMA_T's result to tf32 while the other CTA's chain runs.
            wtT.wait();   // MMA_T
            if (ci + kStep < nchunks) stage_v(ci + kStep);     // the Minv^T region is free now
            dt_to_tf32<false>(t, nullptr);
            // The state after chunk ci - 1 (the other CTA's) arrives; chunk 0
            // starts from the initial state in the TMEM master.
            if (ci > 0) wrx.wait();
            state_pass(t, esc_prev, ci > 0, fb, t.s_gh0[qrow] + t.s_gh1[qrow], s_rxesc);
            publish();
            if (tid == kIssuer1) {
                mma1_part<0>(t, s_bar1);
                mma1_part<1>(t, s_bar1);
            }
        }
        wt1.wait();   // MMA1
        if (tid == kStager) {
            if (ci + kStep < nchunks) stage_qkz(ci + kStep);   // the S^T region is free now
            // this chunk's gate tile into the upper half of the L region
            ++*s_ng;
            ptx::mbar_arrive_expect_tx(s_gbar, C * D * 4);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                ptx::tma_load_4d(sm + OFF_OG + j * kOGBox, &maps.g, j * 32, h, tb0 + t0, bmap, s_gbar);
        }

        // X epilogue (under the levels) into the lower half of the L region
        // (free since MMA1).
        if ((warp & 3) < 2) x_epilogue(t, t.s_beta, OFF_L);
        if constexpr (!RELAY) {
            publish();
            wtT.wait();   // MMA_T
            if (ci + kStep < nchunks) stage_v(ci + kStep);     // the Minv^T region is free now
            dt_to_tf32<false>(t, nullptr);
        }
        publish();

        if (tid == 0) mma2(t, OFF_L, s_bar2);
        // Under MMA2: the gate pass.  The output epilogue (lane quadrants 2,
        // 3) reads rows written by every warp, so it syncs on named barrier 4,
        // on which the U-operand warps (quadrants 0, 1) only arrive: their own
        // path to MMA3 does not wait for the O rows.
        wgate.wait();
        gate_pass(t, OFF_OG);
        if ((warp & 3) < 2) named_barrier_arrive(4, kThreads);
        else named_barrier_sync(4, kThreads);
        wt2.wait();   // MMA2

        // F and the output epilogue, as two independent groups of 8 warps
        // (named barriers): the U rows (lane quadrants 0, 1) write MMA3's U
        // operand and thread 0 issues MMA3 as soon as that group is done; the
        // O_pre rows (quadrants 2, 3) normalise, gate and store o.
        const bool direct = io.cu_seqlens != nullptr && n < C;
        if ((warp & 3) < 2) u_operand_mma3(t, OFF_R, s_bar3);
        else out_epilogue(t, OFF_OG, p.rms_eps, n, direct, io.o + ((rowbase + t0) * H + h) * D, (size_t)H * D, maps,
                          h, tb0 + t0, bmap);
        wt3.wait();   // MMA3

        // S_new = e^{G_last - rho_R} M: the scale is carried in a register and
        // applied by the next chunk's state pass (or the final write-back).
        {
            const float gl = t.s_gh0[qrow] + t.s_gh1[qrow];
            esc_prev = __expf(fb ? 0.f : 0.5f * gl);   // e^{G_last - rho_R}
        }
        if (RELAY && ci + 1 < nchunks) {
            // The master after this chunk and its pending scale e^{G_last -
            // rho_R} to the other CTA, once its region is free (row qrow, the
            // columns of this group; the group-0 threads send the scale).
            uint32_t sv[32];
            tc::ld32(tc::taddr(t.tm, warp, TM_S + grp * 32), sv);
            wfree.wait();
            tc::wait_ld();
            if (!*(volatile int*)s_dead && !(io.drop_relay && ci == 0)) {
                const uint32_t rb = peer_st + (uint32_t)qrow * 512;
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    ptx::st_async_v4(rb + ((uint32_t)(grp * 8 + (q4 ^ (qrow & 7))) << 4), sv[4 * q4], sv[4 * q4 + 1],
                                     sv[4 * q4 + 2], sv[4 * q4 + 3], peer_full);
                if (grp == 0) ptx::st_async_b32(peer_esc + (uint32_t)qrow * 4, __float_as_uint(esc_prev), peer_full);
            }
        }
        // A bounded wait that gave up anywhere in the CTA ends the walk for
        // every thread at once (the vote is uniform).
        tc::fence_before();
        const bool stop = __syncthreads_or(*(volatile int*)s_dead) != 0;
        tc::fence_after();
        if (stop) break;
    }
    const bool dead = __syncthreads_or(*(volatile int*)s_dead) != 0;

    // Final state and conv window back to global memory (not after a give-up:
    // S and the window then keep their old contents; in relay launches by the
    // CTA that ran the last chunk).
    const bool owns_end = !RELAY || (nchunks > 0 && (nchunks - 1) % 2 == role);
    if (!dead && owns_end)
        state_window_out(t, io.S + (size_t)bh * D * D, esc_prev, xg - t.cp, rowbase, T, HD, win, cw.gcp);
    if (tid == kOStore) ptx::bulk_wait_all();
    if (dead) {
        // Give-up path: let everything this CTA issued finish (each wait
        // bounded) before its TMEM and shared memory are released.  The three
        // MMA issuers commit their MMAs to one barrier; the last input-tile and
        // gate-tile phases that were issued are waited for as well.
        if (tid == 0 || tid == kIssuer1 || tid == kIssuerB) tc::commit(s_drain);
        if (tid == kStager) {
            if (*s_nt > 0) ptx::mbar_wait_timed(s_tbar, (uint32_t)((*s_nt - 1) & 1));
            if (*s_ng > 0) ptx::mbar_wait_timed(s_gbar, (uint32_t)((*s_ng - 1) & 1));
        }
        if (tid == 0) ptx::mbar_wait_timed(s_drain, 0);
        // Relay: a state this CTA announced it could take may still be on
        // its way into its shared memory.
        if (RELAY && tid == 0 && nrx > 0) ptx::mbar_wait_timed(s_rxfull, (uint32_t)((nrx - 1) & 1));
    }
    // Relay: neither CTA leaves while the other may still address its
    // shared memory (every wait before this point is bounded, so both get here).
    if constexpr (RELAY) ptx::cluster_sync();
    sync_tc();
    if (warp == 0) tc::dealloc(t.tm, 512);
}

// ---------------------------------------------------------------------------
// Split schedule (few sequence-heads): producer CTAs build the
// state-independent operands of every chunk in parallel and pass them, through
// a ring of slots in the caller's workspace, to one consumer CTA per
// (sequence, head), which keeps the state in TMEM and runs only the chain
// (state pass, MMA1, X epilogue, MMA2, U operand, MMA3, output epilogue).
// All CTAs of the launch are resident at once (cooperative launch).  Each
// producer takes every nprod-th item of the chunk-major list (chunk c of head
// h is item c * heads + h) in increasing order and waits for a free slot only
// at an item's start, when it holds no unpublished item: the lowest
// unfinished item then always finishes (what it waits for belongs to lower
// items), so the schedule makes progress.  Every wait on another CTA is also
// bounded, so a lost item ends as a timeout, not a hang.
// ---------------------------------------------------------------------------
constexpr int kRing = 4;   // slots per head
// A slot: L (tf32, SW128 as in shared memory), V (fp32, SW128), DT and R^T
// (the TMEM images, see img_at), then beta[64], G_last[128] and the fallback flag.
constexpr uint32_t SL_L = 0, SL_V = 65536, SL_DT = 98304, SL_RT = 131072, SL_SMALL = 163840;
constexpr uint32_t kSmallBytes = 1024;
constexpr uint32_t kSlotBytes = SL_SMALL + kSmallBytes;
// Consumer shared memory: the S^T operand, after MMA1 the Diag(beta) X
// operand (lower half) and the U operand (upper half); L; the gate / o tile
// in the R region; V; the small records (two, by chunk parity) in the Minv^T region.
constexpr uint32_t CON_X = OFF_ST, CON_U = OFF_ST + 32768, CON_OG = OFF_R, CON_SMALL = OFF_MT;
// The consumer's operand copies come from warp 14 (lane quadrant 2: idle in
// the X epilogue, so a wait for the next chunk's slot does not hold up the chain).
constexpr int kCStager = 448;

struct SplitIO {
    uint8_t* ring;   // [heads][kRing] slots of kSlotBytes
    int* ready;      // [heads][kRing]: 1 + the chunk a slot holds (0: none yet)
    int* consumed;   // [heads]: chunks whose slot its consumer has read
    int heads;       // sequence-heads of the launch: bh = head0 + [0, heads); CTAs [0, heads) consume
    int head0;
    int nprod;       // producer CTAs: [heads, heads + nprod)
    int drop;        // test injection: producers skip publishing their first item
};

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until *flag >= target (acquire), bounded like the mbarrier waits; a
// give-up marks the CTA dead and records the error.  Skipped in a dead CTA.
__device__ __forceinline__ bool flag_wait(const int* flag, int target, int* dead, int* err) {
    if (*(volatile int*)dead) return false;
    if (ld_acquire(flag) >= target) return true;
    const unsigned long long t0 = ptx::globaltimer_ns();
    for (unsigned i = 1;; ++i) {
        __nanosleep(100);
        if (ld_acquire(flag) >= target) return true;
        if ((i & 15) == 0 && (*(volatile int*)dead || ptx::globaltimer_ns() - t0 > ptx::kWaitLimitNs)) {
            *(volatile int*)dead = 1;
            atomicOr(err, ptx::kErrPrefillWait);
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_split_kernel(const LayerParams p, const PrefillIO io, int* err, const __grid_constant__ Maps maps,
                         const SplitIO sp) {
    extern __shared__ __align__(1024) uint8_t sm[];
    Thr t = make_thr(sm);
    uint64_t* s_bar = reinterpret_cast<uint64_t*>(sm + kBarOff);   // producer: MMA0 done
    uint64_t* s_tbar = s_bar + 1;                                 // producer: input tiles landed
    uint64_t* s_gbar = s_bar + 2;                                 // consumer: gate tile landed
    uint64_t* s_tbarT = s_bar + 3;                                // producer: MMA_T done
    uint64_t* s_bar1 = s_bar + 4;                                 // consumer: MMA1 done
    uint64_t* s_drain = s_bar + 5;                                // give-up path: MMA issuers drained
    uint64_t* s_bar2 = s_bar + 6;                                 // consumer: MMA2 done
    uint64_t* s_bar3 = s_bar + 7;                                 // consumer: MMA3 done
    uint64_t* s_ldA = s_bar + 8;                                  // consumer: L and small record landed
    uint64_t* s_ldV = s_bar + 9;                                  // consumer: V landed
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_bar + 10);
    int* s_dead = reinterpret_cast<int*>(s_tmem + 1);
    int* s_nt = s_dead + 1;   // phases issued: input tiles (producer) or gate tiles (consumer)
    int* s_na = s_dead + 2;   // consumer: L phases issued
    int* s_nv = s_dead + 3;   // consumer: V phases issued

    const int tid = t.tid, warp = t.warp;
    const bool prod = (int)blockIdx.x >= sp.heads;
    const int H = p.H, T = io.T;
    const size_t HD = (size_t)H * D, HD3 = 3 * HD;
    const int nchunks = (T + C - 1) / C;

    if (warp == 0) tc::alloc(s_tmem, 512);
    if (tid == 0) {
        ptx::mbar_init(s_bar, 1);
        ptx::mbar_init(s_tbar, 1);
        ptx::mbar_init(s_gbar, 1);
        ptx::mbar_init(s_tbarT, 1);
        ptx::mbar_init(s_bar1, 1);
        ptx::mbar_init(s_drain, 2);
        ptx::mbar_init(s_bar2, 1);
        ptx::mbar_init(s_bar3, 1);
        ptx::mbar_init(s_ldA, 1);
        ptx::mbar_init(s_ldV, 1);
        ptx::fence_mbar_init();
        *s_dead = 0;
        *s_nt = 0;
        *s_na = 0;
        *s_nv = 0;
    }
    sync_tc();
    t.tm = *s_tmem;

    if (prod) {
        // ---- Producer: items it = c * heads + hh, this CTA's every nprod-th.
        const int total = sp.heads * nchunks;
        Waiter wt{s_bar, s_dead, err, 0u};
        Waiter wtma{s_tbar, s_dead, err, 0u};
        Waiter wtT{s_tbarT, s_dead, err, 0u};
        auto coords = [&](int it, int& hh, int& ci, int& b, int& h) {
            hh = it % sp.heads;
            ci = it / sp.heads;
            const int bh = sp.head0 + hh;
            b = bh / H;
            h = bh - b * H;
        };
        auto stage_qkz = [&](int it) {
            if (tid == kStager) {
                int hh, ci, b, h;
                coords(it, hh, ci, b, h);
                ++*s_nt;
                ptx::mbar_arrive_expect_tx(s_tbar, kStageBytes);
                ptx::tma_load_4d(sm + STG_Q, &maps.q, 0, h, ci * C, b, s_tbar);
                ptx::tma_load_4d(sm + STG_K, &maps.k, 0, h, ci * C, b, s_tbar);
                ptx::tma_load_4d(sm + STG_Z, &maps.z, 0, h, ci * C, b, s_tbar);
                ptx::tma_prefetch_4d(&maps.v, 0, h, ci * C, b);
            }
        };
        auto stage_v = [&](int it) {
            if (tid == 0) {
                int hh, ci, b, h;
                coords(it, hh, ci, b, h);
                ptx::tma_load_4d(sm + STG_V, &maps.v, 0, h, ci * C, b, s_tbar);
            }
        };
        int it = (int)blockIdx.x - sp.heads;
        if (it < total) {
            stage_qkz(it);
            stage_v(it);
        }
        bool first = true;
        for (; it < total; it += sp.nprod) {
            int hh, ci, b, h;
            coords(it, hh, ci, b, h);
            const int t0 = ci * C, n = min(C, T - t0);
            const size_t rowbase = (size_t)b * T;
            uint8_t* slot = sp.ring + ((size_t)hh * kRing + ci % kRing) * kSlotBytes;
            const ConvW cw = conv_consts(t, p, h, HD);
            const float blog = tid < n ? io.beta_logit[(rowbase + t0 + tid) * H + h] : 0.f;
            // The slot is free once its consumer has read the chunk kRing before.
            if (tid == 0 && ci >= kRing && flag_wait(sp.consumed + hh, ci - kRing + 1, s_dead, err))
                fence_proxy_async_global();
            wtma.wait();
            const uint16_t* xg = (t.grp == 0 ? io.q : (t.grp == 1 ? io.k : io.v)) + (size_t)h * D + t.cp;
            const bool big = conv_decay(t, cw, n, ci > 0 ? kWinInputs : kWinState, 0, false, xg,
                                        rowbase + (size_t)t0 - 3, HD, io.conv_state + (size_t)b * 3 * HD3);
            ptx::fence_proxy_async_smem();   // V: source of the bulk store below
            const bool fb = __syncthreads_or(big) != 0;
            const bool live = !*(volatile int*)s_dead;
            if (tid == kStager) {
                if (live) {
                    ptx::bulk_s2g(slot + SL_V, sm + OFF_V, 32768);
                    ptx::bulk_commit();
                }
                if (it + sp.nprod < total) stage_qkz(it + sp.nprod);   // the staging region is free
            }
            norms(t, n, blog, p.l2_eps);
            publish();
            if (fb) exact_fallback(t);
            if (live) lr_build<true>(t, fb, reinterpret_cast<float*>(slot + SL_RT));
            else lr_build<false>(t, fb, nullptr);
            publish();
            if (tid == kStager && live) {
                ptx::bulk_s2g(slot + SL_L, sm + OFF_L, 65536);
                ptx::bulk_commit();
            }
            if (!fb && tid == 0) mma0(t, s_bar);
            if (!fb) wt.wait();   // MMA0
            c1_pass(t);
            tc::wait_st();
            sync_tc();
            inverse_mma_t(t, s_tbarT);
            wtT.wait();   // MMA_T
            if (it + sp.nprod < total) stage_v(it + sp.nprod);   // the Minv^T region is free
            if (live) {
                dt_to_tf32<true>(t, reinterpret_cast<float*>(slot + SL_DT));
                float* small = reinterpret_cast<float*>(slot + SL_SMALL);
                if (tid < C) small[tid] = t.s_beta[tid];
                if (tid < D) small[C + tid] = t.s_gh0[tid] + t.s_gh1[tid];
                if (tid == 0) reinterpret_cast<int*>(small)[C + D] = fb ? 1 : 0;
            }
            if (tid == kStager) ptx::bulk_wait_all();   // L and V written, their smem reads done
            tc::fence_before();
            const bool stop = __syncthreads_or(*(volatile int*)s_dead) != 0;
            tc::fence_after();
            if (stop) break;
            if (tid == kStager && !(sp.drop && first)) {
                fence_proxy_async_global();
                __threadfence();
                st_release(sp.ready + hh * kRing + ci % kRing, ci + 1);
            }
            first = false;
        }
        if (*(volatile int*)s_dead) {
            // Give-up path: MMAs and the tile phases this CTA issued finish
            // (bounded) before its TMEM and shared memory are released.
            if (tid == 0 || tid == kIssuerB) tc::commit(s_drain);
            if (tid == kStager) {
                ptx::bulk_wait_all();
                if (*s_nt > 0) ptx::mbar_wait_timed(s_tbar, (uint32_t)((*s_nt - 1) & 1));
            }
            if (tid == 0) ptx::mbar_wait_timed(s_drain, 0);
        }
    } else {
        // ---- Consumer of sequence-head bh: the chain over its chunks.
        const int hh = (int)blockIdx.x, bh = sp.head0 + hh;
        const int b = bh / H, h = bh - b * H;
        const size_t rowbase = (size_t)b * T;
        Waiter wA{s_ldA, s_dead, err, 0u};
        Waiter wV{s_ldV, s_dead, err, 0u};
        Waiter wgate{s_gbar, s_dead, err, 0u};
        Waiter wt1{s_bar1, s_dead, err, 0u};
        Waiter wt2{s_bar2, s_dead, err, 0u};
        Waiter wt3{s_bar3, s_dead, err, 0u};
        auto slot_of = [&](int ci) { return sp.ring + ((size_t)hh * kRing + ci % kRing) * kSlotBytes; };
        auto load_a = [&](int ci) {   // L and the small record of chunk ci
            const uint8_t* s = slot_of(ci);
            ++*s_na;
            ptx::mbar_arrive_expect_tx(s_ldA, 65536 + kSmallBytes);
            ptx::bulk_g2s(sm + OFF_L, s + SL_L, 65536, s_ldA);
            ptx::bulk_g2s(sm + CON_SMALL + (ci & 1) * kSmallBytes, s + SL_SMALL, kSmallBytes, s_ldA);
        };
        auto load_v = [&](int ci) {
            ++*s_nv;
            ptx::mbar_arrive_expect_tx(s_ldV, 32768);
            ptx::bulk_g2s(sm + OFF_V, slot_of(ci) + SL_V, 32768, s_ldV);
        };
        auto load_gate = [&](int ci) {
            ++*s_nt;
            ptx::mbar_arrive_expect_tx(s_gbar, C * D * 4);
#pragma unroll
            for (int j = 0; j < 4; ++j) ptx::tma_load_4d(sm + CON_OG + j * kOGBox, &maps.g, j * 32, h, ci * C, b, s_gbar);
            if (ci + 1 < nchunks) {   // the next chunk's gate tile into L2 a chunk ahead
#pragma unroll
                for (int j = 0; j < 4; ++j) ptx::tma_prefetch_4d(&maps.g, j * 32, h, (ci + 1) * C, b);
            }
        };
        if (tid < D) t.s_gam[tid] = 0.5f * p.gamma[h * D + tid];
        bool have_next = false;   // stager: the next chunk's slot is published (and its loads issued)
        if (tid == kCStager) {
            load_gate(0);
            if (flag_wait(sp.ready + hh * kRing, 1, s_dead, err)) {
                fence_proxy_async_global();
                load_a(0);
                load_v(0);
            }
        }
        state_in(t, io.S + (size_t)bh * D * D);
        sync_tc();   // the stager's acquire of chunk 0 comes before every thread's reads of its slot
        // DT and R^T of a chunk: loaded into registers while MMA2 of the chunk
        // before runs, written into TMEM once MMA3 of that chunk has completed
        // (DT could go after MMA2, but then the U-operand warps would wait for
        // these loads before their part of the chain: 0.309 -> 0.300 ms on
        // B=1, H=32, T=4096 with both stores after MMA3).
        uint4 dtr[4], rtr[4];
        auto load_dtrt = [&](int cj) {
            const float* dti = reinterpret_cast<const float*>(slot_of(cj) + SL_DT);
            const float* rti = reinterpret_cast<const float*>(slot_of(cj) + SL_RT);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dtr[k] = *reinterpret_cast<const uint4*>(dti + img_at(t, k));
                rtr[k] = *reinterpret_cast<const uint4*>(rti + img_at(t, k));
            }
        };
        auto store_tm = [&](const uint4 (&r)[4], int col) {
            uint32_t v[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) { v[4 * k] = r[k].x; v[4 * k + 1] = r[k].y; v[4 * k + 2] = r[k].z; v[4 * k + 3] = r[k].w; }
            tc::st16(tc::taddr(t.tm, warp, col + t.grp * 16), v);
        };
        load_dtrt(0);
        store_tm(dtr, TM_DT);
        store_tm(rtr, TM_RT);
        float esc_prev = 1.0f;
        for (int ci = 0; ci < nchunks; ++ci) {
            const int t0 = ci * C, n = min(C, T - t0);
            const float* small = reinterpret_cast<const float*>(sm + CON_SMALL + (ci & 1) * kSmallBytes);
            wA.wait();   // L and the small record
            const bool fb = reinterpret_cast<const int*>(small)[C + D] != 0;
            const float gl = small[C + t.qrow];
            state_pass(t, esc_prev, false, fb, gl, nullptr);
            publish();   // S^T operand, rescaled master
            if (tid == kIssuer1) {
                mma1_part<0>(t, s_bar1);
                mma1_part<1>(t, s_bar1);
            }
            // under MMA1: the gate tile becomes gamma sigmoid(gate) (warps 1..15)
            wgate.wait();
            gate_pass(t, CON_OG);
            // under MMA1: is the next chunk published?
            if (tid == kCStager)
                have_next = ci + 1 < nchunks && flag_wait(sp.ready + hh * kRing + (ci + 1) % kRing, ci + 2, s_dead, err);
            wt1.wait();   // MMA1: L and S^T are free
            if (tid == kCStager && have_next) {
                fence_proxy_async_global();
                load_a(ci + 1);
            }
            wV.wait();   // V
            if ((warp & 3) < 2) x_epilogue(t, small, CON_X);
            publish();
            if (tid == kCStager) {
                // every read of chunk ci's slot is done: its producer may refill it
                st_release(sp.consumed + hh, ci + 1);
                if (have_next) load_v(ci + 1);
            }
            if (tid == 0) mma2(t, CON_X, s_bar2);
            const bool more = ci + 1 < nchunks;
            if (more) load_dtrt(ci + 1);   // its slot was acquired before the barrier above
            wt2.wait();   // MMA2
            if ((warp & 3) < 2) u_operand_mma3(t, CON_U, s_bar3);
            else out_epilogue(t, CON_OG, p.rms_eps, n, false, nullptr, 0, maps, h, t0, b);
            wt3.wait();   // MMA3
            if (more) {
                store_tm(dtr, TM_DT);
                store_tm(rtr, TM_RT);
            }
            esc_prev = __expf(fb ? 0.f : 0.5f * gl);   // e^{G_last - rho_R}
            tc::fence_before();
            const bool stop = __syncthreads_or(*(volatile int*)s_dead) != 0;
            tc::fence_after();
            if (stop) break;
            if (tid == kOStore) {
                ptx::bulk_wait_read_all();   // the o tile has left shared memory
                if (ci + 1 < nchunks) load_gate(ci + 1);
            }
        }
        const bool dead = __syncthreads_or(*(volatile int*)s_dead) != 0;
        if (!dead) {
            const uint16_t* x = t.grp == 0 ? io.q : (t.grp == 1 ? io.k : io.v);
            const ConvW cw = conv_consts(t, p, h, HD);
            state_window_out(t, io.S + (size_t)bh * D * D, esc_prev, x + (size_t)h * D, rowbase, T, HD,
                             io.conv_state + (size_t)b * 3 * HD3, cw.gcp);
        }
        if (tid == kOStore) ptx::bulk_wait_all();
        if (dead) {
            if (tid == 0 || tid == kIssuer1) tc::commit(s_drain);
            if (tid == kCStager) {
                if (*s_na > 0) ptx::mbar_wait_timed(s_ldA, (uint32_t)((*s_na - 1) & 1));
                if (*s_nv > 0) ptx::mbar_wait_timed(s_ldV, (uint32_t)((*s_nv - 1) & 1));
                if (*s_nt > 0) ptx::mbar_wait_timed(s_gbar, (uint32_t)((*s_nt - 1) & 1));
            }
            if (tid == 0) ptx::mbar_wait_timed(s_drain, 0);
        }
    }
    sync_tc();
    if (warp == 0) tc::dealloc(t.tm, 512);
}

// Per-device flag: the kernels' attributes are set (the call is idempotent,
// so two host threads setting it at once is harmless).
std::atomic<bool> g_attr_done[64];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// [B][T][H][d] tensor seen as 4-D (d, H, T, B); boxes of `bd` channels of one
// head x 64 tokens.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int H, int T,
              int B, int bd = D, CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize,
                                   (cuuint64_t)T * H * D * esize};
    const cuuint32_t box[4] = {(cuuint32_t)bd, 1, (cuuint32_t)C, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Heads that would leave SMs idle as single CTAs: all of them when twice
// their number fits on the SMs (few-head workloads: otherwise most SMs
// idle), else the heads of a last, partial wave when it fills at most half
// of the SMs; none for single-chunk sequences.  They run on the split
// schedule when the caller gives its workspace, else as relay pairs.  (Packed
// calls, whose lengths only the device knows, use relay pairs for all their
// sequence-heads when twice their number fits, else none; see launch_prefill.)
long long relay_heads(long long heads, int nchunks, int sm_count) {
    if (nchunks < 2 || sm_count < 2) return 0;
    if (2 * heads <= sm_count) return heads;
    const long long rem = heads % sm_count;
    return (rem > 0 && 2 * rem <= sm_count) ? rem : 0;
}

// Workspace of the split schedule for `heads` sequence-heads: the ready and
// consumed flags, then the slots (1 KiB aligned).
size_t split_flag_bytes(long long heads) { return ((size_t)heads * (kRing + 1) * sizeof(int) + 1023) & ~size_t(1023); }
size_t split_bytes(long long heads) { return split_flag_bytes(heads) + (size_t)heads * kRing * kSlotBytes; }

cudaError_t set_attrs(int device) {
    if (device >= 0 && device < 64 && g_attr_done[device].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kda_prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kda_prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kda_prefill_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess && device >= 0 && device < 64) g_attr_done[device].store(true, std::memory_order_release);
    return e;
}

}  // namespace

long long prefill_relay_heads(long long heads, int T, int sm_count) {
    return relay_heads(heads, (T + C - 1) / C, sm_count);
}

size_t prefill_workspace_bytes(int H, int B, int T, const DeviceInfo& dev) {
    const long long rh = relay_heads((long long)B * H, (T + C - 1) / C, dev.sm_count);
    return rh > 0 && rh < dev.sm_count ? split_bytes(rh) : 0;
}

cudaError_t launch_prefill(const LayerParams& p, const PrefillIO& io, const DeviceInfo& dev,
                           int* err_word, cudaStream_t stream) {
    const long long grid = (long long)io.B * p.H;
    if (grid <= 0 || io.T <= 0) return cudaSuccess;
    if (cudaError_t e = set_attrs(dev.device); e != cudaSuccess) return e;
    Maps maps;
    const int mB = io.cu_seqlens ? 1 : io.B;   // packed sequences: one token axis of length io.T
    if (!make_map(&maps.q, io.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.H, io.T, mB) ||
        !make_map(&maps.k, io.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.H, io.T, mB) ||
        !make_map(&maps.v, io.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.H, io.T, mB) ||
        !make_map(&maps.z, io.z, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.H, io.T, mB) ||
        !make_map(&maps.g, io.gate_logit, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.H, io.T, mB, 32,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&maps.o, io.o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.H, io.T, mB, 32,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int nchunks = (io.T + C - 1) / C;
    // Packed sequences (their lengths are on the device): relay pairs for all
    // sequence-heads when twice their number fits on the SMs, else none.
    const long long rh = io.cu_seqlens ? (2 * grid <= dev.sm_count ? grid : 0)
                                       : relay_heads(grid, nchunks, dev.sm_count);
    const long long single = grid - rh;
    const bool split = rh > 0 && rh < dev.sm_count && io.workspace != nullptr && io.workspace_bytes >= split_bytes(rh);
    if (single > 0) {
        PrefillIO io1 = io;
        io1.head0 = 0;
        kda_prefill_kernel<false><<<(unsigned)single, kThreads, kSmemBytes, stream>>>(p, io1, err_word, maps);
        count_launches(1);
        if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
    }
    if (rh > 0 && split) {
        // The heads [single, grid) on the split schedule: one consumer CTA per
        // head and the rest of the SMs as producers, all resident at once.
        SplitIO sp;
        uint8_t* ws = static_cast<uint8_t*>(io.workspace);
        sp.ready = reinterpret_cast<int*>(ws);
        sp.consumed = sp.ready + rh * kRing;
        sp.ring = ws + split_flag_bytes(rh);
        sp.heads = (int)rh;
        sp.head0 = (int)single;
        sp.nprod = (int)std::min<long long>(dev.sm_count - rh, rh * nchunks);
        sp.drop = io.drop_split;
        if (cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)rh * (kRing + 1) * sizeof(int), stream); e != cudaSuccess)
            return e;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)(rh + sp.nprod));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = io.nofit_split ? cudaErrorCooperativeLaunchTooLarge
                                       : cudaLaunchKernelEx(&cfg, kda_prefill_split_kernel, p, io, err_word, maps, sp);
        if (e == cudaSuccess) {
            count_launches(1);
            return cudaGetLastError();
        }
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        // The launch cannot be resident all at once on the device as this
        // process sees it (fewer SMs than the device has): the same heads run
        // as relay pairs instead, with the same results.
        (void)cudaGetLastError();
    }
    if (rh > 0) {
        // The heads [single, grid) as CTA pairs, each pair one cluster of two
        // (scheduled together; a pair waits on nothing outside itself).
        PrefillIO io2 = io;
        io2.head0 = (int)single;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)(2 * rh));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, kda_prefill_kernel<true>, p, io2, err_word, maps);
        count_launches(1);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace kda
