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
//         on the TMEM master M = Diag(e^rho) S0; S_new = e^{G_last-rho} M, that
//         row scale being applied by the next chunk's pass over the master.
// The unit-lower inverse is a forward substitution on CUDA cores for the
// diagonal 16 x 16 blocks and warp-level tf32 MMAs for the rest.
#include <cuda.h>
#include <cudaTypedefs.h>

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

// 16 warps: warp w reaches TMEM lanes [32 (w % 4), +32) and takes column group
// w / 4 of every TMEM pass; in the thread-per-channel passes the same thread
// owns channel c = its TMEM lane and group grp = w / 4.
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
    float* s_beta = reinterpret_cast<float*>(sm + OFF_SMALL);   // [64]
    float* s_rq = s_beta + 64;                                    // [64]
    float* s_rk = s_rq + 64;                                      // [64]
    float* s_part = s_rk + 64;                                    // [4][64] RMS partial sums
    float* s_gh0 = s_part + 256;                                  // [128] decay sum over tokens 0..31
    float* s_gh1 = s_gh0 + 128;                                   // [128] decay sum over tokens 32..63
    float* s_gam = s_gh1 + 128;                                   // [128] gamma / 2 of this head
    float* s_win = reinterpret_cast<float*>(sm + OFF_WIN);        // [2][3][3][128], by chunk parity
    // mbarriers.  Each completes at most one phase per chunk and every thread
    // that waits on one waits on it once per chunk, so no waiter can fall two
    // phases behind (a parity wait would then alias onto a later phase).
    uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_gam + 128);   // MMA0 done
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

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    const int qrow = (warp & 3) * 32 + lane;   // TMEM lane; channel of the per-channel passes
    const int grp = warp >> 2;                  // column group / per-channel role (0..3)
    const int c = qrow;

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
    if (tid < D) s_gam[tid] = 0.5f * p.gamma[h * D + tid];   // gamma sigmoid(g) = s_gam + s_gam tanh(g / 2)
    sync_tc();
    // Relay pairs: the other CTA's barriers are initialised before either
    // CTA touches them (both CTAs of a cluster are scheduled together).
    if constexpr (RELAY) ptx::cluster_sync();
    const uint32_t tm = *s_tmem;
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

    // Initial state into the TMEM master (row qrow, columns of this group).
    {
        const float* src = io.S + ((size_t)bh * D + qrow) * D + grp * 32;
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 v = *reinterpret_cast<const float4*>(src + j);
            r[j] = __float_as_uint(v.x); r[j + 1] = __float_as_uint(v.y);
            r[j + 2] = __float_as_uint(v.z); r[j + 3] = __float_as_uint(v.w);
        }
        tc::st32(tc::taddr(tm, warp, TM_S + grp * 32), r);
        tc::wait_st();
    }

    // Conv / decay roles: grp 0, 1, 2 = conv of q, k, v; grp 3 = decay; each
    // thread takes the channel pair (cp, cp + 1) for tokens [32 th, 32 th + 32).
    float* win = io.conv_state + (size_t)b * 3 * HD3;
    const int cp = (tid & 63) * 2;
    const int th = (tid >> 6) & 1;
    const size_t gcp = (size_t)(grp < 3 ? grp : 0) * HD + (size_t)h * D + cp;
    f32x2 W0 = 0, W1 = 0, W2 = 0, W3 = 0;   // taps (tap 3 multiplies the current token)
    f32x2 nEA = 0, DTB = 0;                 // -exp(A_log), dt_bias
    if (grp < 3) {
        const float4 a = *reinterpret_cast<const float4*>(p.conv_w + gcp * 4);
        const float4 bq = *reinterpret_cast<const float4*>(p.conv_w + (gcp + 1) * 4);
        // taps halved: the conv then yields x / 2, the argument SiLU takes
        W0 = pk(0.5f * a.x, 0.5f * bq.x); W1 = pk(0.5f * a.y, 0.5f * bq.y);
        W2 = pk(0.5f * a.z, 0.5f * bq.z); W3 = pk(0.5f * a.w, 0.5f * bq.w);
        if (th == 0) {
#pragma unroll
            for (int j = 0; j < 3; ++j)
                *reinterpret_cast<float2*>(s_win + (grp * 3 + j) * D + cp) =
                    *reinterpret_cast<const float2*>(win + j * HD3 + gcp);
        }
    } else {
        nEA = pk(-expf(p.A_log[h * D + cp]), -expf(p.A_log[h * D + cp + 1]));
        DTB = pk(p.dt_bias[h * D + cp], p.dt_bias[h * D + cp + 1]);
    }
    // Swizzled addressing of the channel pair as the K index of the L
    // (128-row) and R / V (64-row) operand layouts.
    const uint32_t kpL = (uint32_t)((cp >> 5) * 128 * 128 + (cp & 3) * 4);
    const uint32_t kpR = (uint32_t)((cp >> 5) * 64 * 128 + (cp & 3) * 4);
    const int pch = (cp >> 2) & 7;

    // Swizzled addressing of channel c as the K index of the L (128-row) and
    // R / V (64-row) operand layouts.
    const uint32_t kcL = (uint32_t)((c >> 5) * 128 * 128 + (c & 3) * 4);
    const uint32_t kcR = (uint32_t)((c >> 5) * 64 * 128 + (c & 3) * 4);
    const int cch = (c >> 2) & 7;

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

    // State pass: the S^T operand of MMA1 scaled by e^{rho_L} to shared
    // memory and the TMEM master scaled by e^{rho_R} (both also by the
    // previous chunk's pending scale).  The state comes from the TMEM master,
    // or (relay launches, after chunk 0) from the rows the other CTA stored
    // into the S^T region, which the operand then overwrites.
    auto state_pass = [&](bool rx, bool fb) {
        uint32_t v[32];
        const int j0 = grp * 32;
        const uint32_t ta = tc::taddr(tm, warp, TM_S + j0);
        if (rx) {
            const uint32_t rb = OFF_ST + (uint32_t)qrow * 512;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const uint4 x = at<uint4>(sm, rb + ((uint32_t)(grp * 8 + (q4 ^ (qrow & 7))) << 4));
                v[4 * q4] = x.x; v[4 * q4 + 1] = x.y; v[4 * q4 + 2] = x.z; v[4 * q4 + 3] = x.w;
            }
            esc_prev = s_rxesc[qrow];
            __syncthreads();   // every received row is read before the operand overwrites it
        } else {
            tc::ld32(ta, v);
            tc::wait_ld();
        }
        const float gl = s_gh0[qrow] + s_gh1[qrow];
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
    };

    // DT -> tf32 in place (A operand of MMA2).
    auto dt_to_tf32 = [&]() {
        uint32_t v[16];
        const uint32_t ta = tc::taddr(tm, warp, TM_DT + grp * 16);
        tc::ld16(ta, v);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = tc::f2tf32(__uint_as_float(v[i]));
        tc::st16(ta, v);
    };

    for (int ci = role; ci < nchunks; ci += kStep) {
        const int t0 = ci * C;
        const int n = min(C, T - t0);

        // ---- A1: conv + SiLU per channel over the chunk (from the staged
        //      tiles); decay and its cumulative sum.  Loads of token group
        //      g + 1 are issued before the stores of group g.
        bool big = false;
        // beta logits of the chunk, consumed after the conv phase.
        const float blog = tid < n ? io.beta_logit[(rowbase + t0 + tid) * H + h] : 0.f;
        wtma.wait();
        if (grp < 3) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(
                sm + (grp == 0 ? STG_Q : (grp == 1 ? STG_K : STG_V))) + (cp >> 1);
            const uint32_t dst = grp == 0 ? OFF_L + kpL + C * 128 : (grp == 1 ? OFF_L + kpL : OFF_V + kpR);
            auto unpk_bf2 = [](uint32_t u) { return pk(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)); };
            f32x2 M3, M2, M1;   // window, oldest first
            if (RELAY && th == 0 && ci > 0) {
                // the chunk before ran in the other CTA: its last three inputs from global memory
                const uint16_t* xg = (grp == 0 ? io.q : (grp == 1 ? io.k : io.v)) + (size_t)h * D + cp;
                const size_t r3 = rowbase + (size_t)t0 - 3;
                M3 = unpk_bf2(*reinterpret_cast<const uint32_t*>(xg + r3 * HD));
                M2 = unpk_bf2(*reinterpret_cast<const uint32_t*>(xg + (r3 + 1) * HD));
                M1 = unpk_bf2(*reinterpret_cast<const uint32_t*>(xg + (r3 + 2) * HD));
            } else if (th == 0) {
                const float* w = s_win + ((ci & 1) * 9 + grp * 3) * D + cp;
                M3 = pk(w[0], w[1]); M2 = pk(w[D], w[D + 1]); M1 = pk(w[2 * D], w[2 * D + 1]);
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
                        f32x2 pre = mul2(W0, M3);
                        pre = fma2(W1, M2, pre);
                        pre = fma2(W2, M1, pre);
                        pre = fma2(W3, x[i], pre);
                        y[i] = silu2_of_half(pre);
                        M3 = M2; M2 = M1; M1 = x[i];
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const bool ok = r0 + g * 8 + i < n;
                        f32x2 pre = mul2(W0, M3);
                        pre = fma2(W1, M2, pre);
                        pre = fma2(W2, M1, pre);
                        pre = fma2(W3, x[i], pre);
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
            if (th == 1) {   // the next chunk's first half starts from this window
                float* w = s_win + (((ci + 1) & 1) * 9 + grp * 3) * D + cp;
                upk(M3, w[0], w[1]);
                upk(M2, w[D], w[D + 1]);
                upk(M1, w[2 * D], w[2 * D + 1]);
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
                    const f32x2 sp = softplus2(add2(zc[i], DTB));
                    if (r0 + g * 8 + i < n) G = fma2(nEA, sp, G);
                    gg[i] = G;
                }
                const uint32_t rb = OFF_R + kpR + (uint32_t)(r0 + g * 8) * 128 + (pch << 4);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    at<f32x2>(sm, (rb ^ (uint32_t)(i << 4)) + i * 128) = gg[i];
                }
            }
            *reinterpret_cast<f32x2*>((th == 0 ? s_gh0 : s_gh1) + cp) = G;
            float ga, gb;
            upk(G, ga, gb);
            big = -ga > 0.5f * kMaxSpan || -gb > 0.5f * kMaxSpan;   // a half beyond kMaxSpan / 2
        }
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

        // ---- A2: per-token norms of the conv outputs (4 threads per row, one
        //      per 32-channel block; the 8 lanes of a quarter warp take 8 rows of
        //      one block, so their 16-byte loads hit 8 different bank groups) and beta.
        {
            const int R = (tid & 7) + 8 * (tid >> 5), part = (tid >> 3) & 3;   // y_k rows 0..63, y_q rows 64..127
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 v = at<float4>(sm, OFF_L + tc::sw128(R, part * 32 + j, 128));
                ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            ss += __shfl_xor_sync(0xffffffffu, ss, 16);
            if (part == 0) (R < C ? s_rk : s_rq)[R & (C - 1)] = rsqrtf(ss + p.l2_eps);
            if (tid < C)
                s_beta[tid] = tid < n ? sigmoidf_(blog) : 0.f;
        }

        // ---- D: state pass (relay launches: later, once the state has arrived).
        if (!RELAY) state_pass(false, fb);
        publish();   // norms, beta; S^T operand and rescaled master

        // ---- A2b (rare): exact [A'; P] when the chunk decays by more than kMaxSpan.
        if (fb) {
            const int R = qrow;                // D0 row: A' rows 0..63, P rows 64..127
            const int r = R & (C - 1);
            const bool isP = R >= C;
            const float rn = isP ? s_rq[r] : s_rk[r];
#pragma unroll 1
            for (int g8 = 0; g8 < 2; ++g8) {
                uint32_t out[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int col = grp * 16 + g8 * 8 + i;
                    float acc = 0.f;
                    if (isP ? col <= r : col < r) {
#pragma unroll 4
                        for (int ch = 0; ch < D; ++ch) {
                            const float a = at<float>(sm, OFF_L + tc::sw128(R, ch, 128));
                            const float gr = at<float>(sm, OFF_R + tc::sw128(r, ch, C)) + (r >= 32 ? s_gh0[ch] : 0.f);
                            const float kk = at<float>(sm, OFF_L + tc::sw128(col, ch, 128));
                            const float gi = at<float>(sm, OFF_R + tc::sw128(col, ch, C)) + (col >= 32 ? s_gh0[ch] : 0.f);
                            acc = fmaf(a * kk, expf(gr - gi), acc);
                        }
                    }
                    out[i] = __float_as_uint(acc * rn * s_rk[col]);
                }
                tc::st8(tc::taddr(tm, warp, TM_D0 + grp * 16 + g8 * 8), out);
            }
            tc::wait_st();
            __syncthreads();
        }

        // ---- A3: L, R (shared memory, in place over the staging) and R^T
        //      (TMEM), channel c, tokens [16 grp, 16 grp + 16), 8 at a time.
        {
            // rho_L = rho_R = G_last / 2, or (0, G_last) on the fallback path
            const float gl = s_gh0[c] + s_gh1[c];
            const float rl = fb ? 0.f : 0.5f * gl, rr = fb ? gl : 0.5f * gl;
            const float goff = grp >= 2 ? s_gh0[c] : 0.f;   // tokens 32..63 add the first half
#pragma unroll 1
            for (int g8 = 0; g8 < 2; ++g8) {
                uint32_t rt[8];
                float g[8], yk[8], yq[8];
                const int r0 = grp * 16 + g8 * 8;
                const float4 nk0 = *reinterpret_cast<const float4*>(s_rk + r0), nk1 = *reinterpret_cast<const float4*>(s_rk + r0 + 4);
                const float4 nq0 = *reinterpret_cast<const float4*>(s_rq + r0), nq1 = *reinterpret_cast<const float4*>(s_rq + r0 + 4);
                const float nk[8] = {nk0.x, nk0.y, nk0.z, nk0.w, nk1.x, nk1.y, nk1.z, nk1.w};
                const float nq[8] = {nq0.x, nq0.y, nq0.z, nq0.w, nq1.x, nq1.y, nq1.z, nq1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = r0 + i;
                    const uint32_t ro = (uint32_t)(r * 128 + ((cch ^ (r & 7)) << 4));
                    g[i] = at<float>(sm, OFF_R + kcR + ro) + goff;
                    yk[i] = at<float>(sm, OFF_L + kcL + ro) * nk[i];
                    yq[i] = at<float>(sm, OFF_L + kcL + C * 128 + ro) * nq[i];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = grp * 16 + g8 * 8 + i;
                    const uint32_t ro = (uint32_t)(r * 128 + ((cch ^ (r & 7)) << 4));
                    const float eL = __expf(g[i] - rl);
                    const float eR = __expf(rr - g[i]);
                    rt[i] = tc::f2tf32(yk[i] * eR);
                    at<uint32_t>(sm, OFF_L + kcL + ro) = tc::f2tf32(yk[i] * eL);
                    at<uint32_t>(sm, OFF_L + kcL + C * 128 + ro) = tc::f2tf32(yq[i] * eL);
                    at<uint32_t>(sm, OFF_R + kcR + ro) = rt[i];
                }
                tc::st8(tc::taddr(tm, warp, TM_RT + grp * 16 + g8 * 8), rt);
            }
        }
        publish();

        // ---- MMA0: [A'; P] = L R^T.
        if (!fb && tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 64);
#pragma unroll 1
            for (int ks = 0; ks < D / 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ss(tm + TM_D0, tc::desc_sw128(ptx::smem_u32(sm + OFF_L + kb * 16384 + kin * 32)),
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_R + kb * 8192 + kin * 32)), id, ks > 0);
            }
            tc::commit(s_bar);
        }

        // ---- MMA1: D1 = L (Diag(e^rho_L) S0) = [K_g S0; Q_g S0] (runs under the
        //      inverse), issued by warp 10 in two halves: K blocks 0, 1 before
        //      C1 and 2, 3 after it (warp 10 has little work in C1 and C2).
        auto mma1_part = [&](int half) {
            constexpr uint32_t id = tc::idesc_tf32(128, 128);
#pragma unroll 1
            for (int ks = half * 8; ks < half * 8 + 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ss(tm + TM_D1,
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_L + kb * 16384 + kin * 32)),
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_ST + kb * 16384 + kin * 32)), id, ks > 0);
            }
            if (half == 1) tc::commit(s_bar1);
        };
        if (!RELAY && tid == kIssuer1) mma1_part(0);
        if (!fb) wt.wait();   // MMA0

        // ---- C1: N = Diag(beta) A' to shared memory as N^T (row b holds
        //      column b of N; 64-row SW128 layout), D0 -> [I; P] in TMEM (row
        //      qrow, columns [16 grp, 16 grp + 16)).
        {
            const bool isA = qrow < C;
            const int r = isA ? qrow : qrow - C;
            const float br = s_beta[r];
            const int i0 = grp * 16;
            uint32_t v[16];
            tc::ld16(tc::taddr(tm, warp, TM_D0 + i0), v);
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
            tc::st16(tc::taddr(tm, warp, TM_D0 + i0), v);
        }
        tc::wait_st();
        sync_tc();

        if (!RELAY && tid == kIssuer1) mma1_part(1);

        // ---- C2: Minv = (I + N)^{-1} (N strictly lower) by 16 x 16 blocks.
        //      Pass 1: forward substitution with the diagonal block I + N_II
        //      on the right-hand sides [I | N_I0 .. N_I(I-1)], giving Minv_II
        //      and E_IK = Minv_II N_IK.  Passes 2..4, level by level
        //      (I - J = 1, 2, 3): Minv_IJ = -sum_{J <= K < I} E_IK Minv_KJ, one
        //      warp per block.  Minv is kept transposed and tf32-rounded in the
        //      SW128 layout of the MMA_T operand (row j holds column j of Minv).
        {
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
                        for (int t = 0; t < 4; ++t)
                            if (4 * q + t > i) x[4 * q + t] = fmaf(-nv[t], x[i], x[4 * q + t]);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {   // tf32-rounded: operands of the level MMAs and of MMA_T
                    const uint4 u = make_uint4(tc::f2tf32(x[4 * q]), tc::f2tf32(x[4 * q + 1]),
                                               tc::f2tf32(x[4 * q + 2]), tc::f2tf32(x[4 * q + 3]));
                    at<uint4>(sm, K < 0 ? MT(I * 16 + cc, I * 16 + q * 4) : EC((I * (I - 1)) / 2 + K, cc, q * 4)) = u;
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
            // Levels, on warps 15, 14, 11 (blocks J = 0, 1, 2), which have no rows
            // in the X epilogue running meanwhile: warp J computes the 16 x 16
            // block Minv_{J+lev, J} with warp-level m16n8k8 tf32 MMAs (operands
            // stored tf32-rounded; the result is rounded once more when stored).
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
#pragma unroll 1
                    for (int ks = 0; ks < C / 8; ++ks) {
                        const int kb = ks >> 2, kin = ks & 3;
                        tc::mma_ts(tm + TM_DT, tm + TM_D0 + ks * 8,
                                   tc::desc_sw128(ptx::smem_u32(sm + OFF_MT + kb * 8192 + kin * 32)), id, ks > 0);
                    }
                    tc::commit(s_tbarT);
                }
            }
        }
        if constexpr (RELAY) {
            // MMA_T's result to tf32 while the other CTA's chain runs.
            wtT.wait();   // MMA_T
            if (ci + kStep < nchunks) stage_v(ci + kStep);     // the Minv^T region is free now
            dt_to_tf32();
            // The state after chunk ci - 1 (the other CTA's) arrives; chunk 0
            // starts from the initial state in the TMEM master.
            if (ci > 0) wrx.wait();
            state_pass(ci > 0, fb);
            publish();
            if (tid == kIssuer1) {
                mma1_part(0);
                mma1_part(1);
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

        // ---- E (lane quadrants 0, 1, under the levels): X = V - K_g S0 ->
        //      Diag(beta) X, the B operand of MMA2 (N = 128 value channels x
        //      2 K blocks of 32 tokens, 16 KiB each) in the lower half of the L
        //      region (free since MMA1); clear D1 top.
        if ((warp & 3) < 2) {
            const int r = qrow;   // token
            const float br = s_beta[r];
            const uint32_t kr = OFF_L + (uint32_t)((r >> 5) * 16384 + grp * 32 * 128 + (r & 3) * 4);
            const int rch = (r >> 2) & 7;
            const uint32_t vrow = OFF_V + r * 128;
            uint32_t v[32];
            const uint32_t ta = tc::taddr(tm, warp, TM_D1 + grp * 32);
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
        if constexpr (!RELAY) {
            publish();
            wtT.wait();   // MMA_T
            if (ci + kStep < nchunks) stage_v(ci + kStep);     // the Minv^T region is free now
            dt_to_tf32();
        }
        publish();

        // ---- MMA2: D1 += [Minv; P Minv] Diag(beta) X = [U; P U] (N = 128: a
        //      tf32 MMA costs about the same per instruction at N = 64 and 128).
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_tf32(128, 128);
#pragma unroll 1
            for (int ks = 0; ks < C / 8; ++ks) {
                const int kb = ks >> 2, kin = ks & 3;
                tc::mma_ts(tm + TM_D1, tm + TM_DT + ks * 8,
                           tc::desc_sw128(ptx::smem_u32(sm + OFF_L + kb * 16384 + kin * 32)), id, 1u);
            }
            tc::commit(s_bar2);
        }
        // Under MMA2: the gate tile becomes gamma * sigmoid(gate) in place, rows
        // spread over warps 1..15 (warp 0 issued MMA2).  The output epilogue
        // (lane quadrants 2, 3) reads rows written by every warp, so it syncs
        // on named barrier 4, on which the U-operand warps (quadrants 0, 1)
        // only arrive: their own path to MMA3 does not wait for the O rows.
        wgate.wait();
        if (warp > 0) {   // lane = (box, 16-byte chunk) of a row: channels 4 lane .. 4 lane + 3
            const int box = lane >> 3, ch = lane & 7;
            const float4 gm = *reinterpret_cast<const float4*>(s_gam + lane * 4);
#pragma unroll 1
            for (int r = warp - 1; r < C; r += 15) {
                const uint32_t o = OFF_OG + box * kOGBox + r * 128 + ((ch ^ (r & 7)) << 4);
                const float4 gv = at<float4>(sm, o);
                at<float4>(sm, o) = make_float4(fmaf(gm.x, tanhf_(0.5f * gv.x), gm.x), fmaf(gm.y, tanhf_(0.5f * gv.y), gm.y),
                                                fmaf(gm.z, tanhf_(0.5f * gv.z), gm.z), fmaf(gm.w, tanhf_(0.5f * gv.w), gm.w));
            }
        }
        if ((warp & 3) < 2) named_barrier_arrive(4, kThreads);
        else named_barrier_sync(4, kThreads);
        wt2.wait();   // MMA2

        // ---- F and the output epilogue, as two independent groups of 8 warps
        //      (named barriers): the U rows (lane quadrants 0, 1) write MMA3's
        //      U operand and thread 0 issues MMA3 as soon as that group is done;
        //      the O_pre rows (quadrants 2, 3) take their sums of squares, then
        //      RMSNorm x gamma sigmoid(gate) -> o, written over the gate tile
        //      and stored by TMA (rows past T clipped by the copy).  The last,
        //      partial chunk of a packed sequence stores its rows < n directly:
        //      the rows after it belong to the next sequence.
        const bool direct = io.cu_seqlens != nullptr && n < C;
        if ((warp & 3) < 2) {
            const int r = qrow;
            const uint32_t kr = (uint32_t)((r >> 5) * 128 * 128 + (r & 3) * 4);
            const int rch = (r >> 2) & 7;
            uint32_t v[32];
            tc::ld32(tc::taddr(tm, warp, TM_D1 + grp * 32), v);
            tc::wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = grp * 32 + jj;
                at<uint32_t>(sm, OFF_R + kr + j * 128 + ((rch ^ (j & 7)) << 4)) = tc::f2tf32(__uint_as_float(v[jj]));
            }
            ptx::fence_proxy_async_smem();
            tc::fence_before();
            named_barrier_sync(2, 256);   // U operand complete
            // ---- MMA3 (overlaps the output epilogue): M += R^T U.
            if (tid == 0) {
                tc::fence_after();
                constexpr uint32_t id = tc::idesc_tf32(128, 128);
#pragma unroll 1
                for (int ks = 0; ks < C / 8; ++ks) {
                    const int kb = ks >> 2, kin = ks & 3;
                    tc::mma_ts(tm + TM_S, tm + TM_RT + ks * 8,
                               tc::desc_sw128(ptx::smem_u32(sm + OFF_R + kb * 16384 + kin * 32)), id, 1u);
                }
                tc::commit(s_bar3);
            }
        } else {
            const int r = qrow - C;
            float ss = 0.f, ss2 = 0.f;
            uint32_t w[32];
            tc::ld32(tc::taddr(tm, warp, TM_D1 + grp * 32), w);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                ss = fmaf(__uint_as_float(w[i]), __uint_as_float(w[i]), ss);
                ss2 = fmaf(__uint_as_float(w[i + 1]), __uint_as_float(w[i + 1]), ss2);
            }
            s_part[grp * C + r] = ss + ss2;
            named_barrier_sync(3, 256);   // the four column groups' partial sums
            const float inv = rsqrtf((s_part[r] + s_part[C + r] + s_part[2 * C + r] + s_part[3 * C + r]) *
                                         (1.0f / D) + p.rms_eps);
            const uint32_t gbase = OFF_OG + grp * kOGBox + r * 128;   // row r of box grp (SW128)
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
                    float* orow = io.o + ((rowbase + t0 + r) * H + h) * D + grp * 32 + g8 * 8;
                    *reinterpret_cast<float4*>(orow) = oa;
                    *reinterpret_cast<float4*>(orow + 4) = ob;
                }
            }
            ptx::fence_proxy_async_smem();
            named_barrier_sync(3, 256);   // the o tile is complete
            if (tid == kOStore && !direct) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    ptx::tma_store_4d(&maps.o, j * 32, h, tb0 + t0, bmap, sm + OFF_OG + j * kOGBox);
                ptx::bulk_commit();
            }
        }
        wt3.wait();   // MMA3
        // the next chunk's conv phase overwrites the tile: its reads must be done
        if (tid == kOStore) ptx::bulk_wait_read_all();

        // S_new = e^{G_last - rho_R} M: the scale is carried in a register and
        // applied by the next chunk's state pass (or the final write-back).
        {
            const float gl = s_gh0[qrow] + s_gh1[qrow];
            esc_prev = __expf(fb ? 0.f : 0.5f * gl);   // e^{G_last - rho_R}
        }
        if (RELAY && ci + 1 < nchunks) {
            // The master after this chunk and its pending scale e^{G_last -
            // rho_R} to the other CTA, once its region is free (row qrow, the
            // columns of this group; the group-0 threads send the scale).
            uint32_t sv[32];
            tc::ld32(tc::taddr(tm, warp, TM_S + grp * 32), sv);
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
    if (!dead && owns_end) {
        float* dst = io.S + ((size_t)bh * D + qrow) * D + grp * 32;
        uint32_t s[32];
        tc::ld32(tc::taddr(tm, warp, TM_S + grp * 32), s);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(esc_prev * __uint_as_float(s[j]), esc_prev * __uint_as_float(s[j + 1]),
                            esc_prev * __uint_as_float(s[j + 2]), esc_prev * __uint_as_float(s[j + 3]));
        // Final window: the last three inputs of the sequence (older taps from
        // the initial window when T < 3).
        if (grp < 3 && th == 0) {
            const uint16_t* x = grp == 0 ? io.q : (grp == 1 ? io.k : io.v);
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int t = T - 3 + j;
                float2 w;
                if (t >= 0) {
                    const uint32_t u = *reinterpret_cast<const uint32_t*>(x + ((rowbase + t) * H + h) * D + cp);
                    w = make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
                } else {   // an older tap of the initial window (not yet overwritten: j + T > j)
                    w = *reinterpret_cast<const float2*>(win + (j + T) * HD3 + gcp);
                }
                *reinterpret_cast<float2*>(win + j * HD3 + gcp) = w;
            }
        }
    }
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
    if (warp == 0) tc::dealloc(tm, 512);
}

// Per-device flag: the kernel's attributes are set (the call is idempotent,
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

// Heads that run as relay pairs: all of them when twice their number fits
// on the SMs (few-head workloads: otherwise most SMs idle), else the heads of
// a last, partial wave when it fills at most half of the SMs (its pairs then
// finish in about half the time of single CTAs); none for single-chunk
// sequences or packed ones.
long long relay_heads(long long heads, int nchunks, int sm_count) {
    if (nchunks < 2 || sm_count < 2) return 0;
    if (2 * heads <= sm_count) return heads;
    const long long rem = heads % sm_count;
    return (rem > 0 && 2 * rem <= sm_count) ? rem : 0;
}

}  // namespace

long long prefill_relay_heads(long long heads, int T, int sm_count) {
    return relay_heads(heads, (T + C - 1) / C, sm_count);
}

size_t prefill_workspace_bytes(int, int, int, const DeviceInfo&) { return 0; }

cudaError_t launch_prefill(const LayerParams& p, const PrefillIO& io, const DeviceInfo& dev,
                           int* err_word, cudaStream_t stream) {
    const long long grid = (long long)io.B * p.H;
    if (grid <= 0 || io.T <= 0) return cudaSuccess;
    if (dev.device < 0 || dev.device >= 64 || !g_attr_done[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kda_prefill_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kda_prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev.device >= 0 && dev.device < 64) g_attr_done[dev.device].store(true, std::memory_order_release);
    }
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
    const long long rh = io.cu_seqlens ? 0 : relay_heads(grid, (io.T + C - 1) / C, dev.sm_count);
    const long long single = grid - rh;
    if (single > 0) {
        PrefillIO io1 = io;
        io1.head0 = 0;
        kda_prefill_kernel<false><<<(unsigned)single, kThreads, kSmemBytes, stream>>>(p, io1, err_word, maps);
        count_launches(1);
        if (cudaError_t e = cudaGetLastError(); e != cudaSuccess) return e;
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
