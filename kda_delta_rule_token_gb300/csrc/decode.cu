// Decode: one KDA token for B sequences in ONE kernel launch.
//
// Follows "Kimi K3 Metal Gap Analysis", section 2 "KDA Attention": rows
// "Conv4 + SiLU", "L2 normalize q/k", "Decay compute", "Recurrence" and "O
// projection" (read-out, head RMSNorm and sigmoid gate), fused the way the
// "Fused KDA token" note of "Metal (Apple GPU) backend for Kimi K3" fuses
// them (one submission per token), laid out for GB300's HBM3e:
//
//  * one CTA of 256 threads per (sequence, head), three CTAs resident per SM
//    (five for the bf16 state);
//  * the 64 KiB fp32 state moves as ONE bulk TMA copy each way
//    (cp.async.bulk global -> shared on an mbarrier, shared -> global as a
//    bulk group), so a whole state is in flight per CTA with one instruction
//    and the load overlaps the conv / norm / decay prologue;
//  * the update runs from shared memory in two passes, keeping registers low
//    enough for three CTAs per SM: warp w owns rows [16w, 16w+16), lane l
//    owns columns [4l, 4l+4) (one 512-byte row per warp access, no bank
//    conflicts);
//  * u = S'^T k and the read-out p = S'^T q come from the same first pass
//    (S' = Diag(e^gk) S); lanes own distinct columns, so column sums need only
//    in-thread adds plus one 8-way shared-memory reduction;
//  * o_pre = S_new^T q = p + (q^.k^) delta with delta = beta (v - u): the
//    read-out needs no extra pass over the state.
//
// The same kernel, instantiated for a bfloat16 state, keeps the state as
// bf16 in memory (32 KiB per head, half the bytes each way): it is widened
// to fp32 as pass 1 and pass 2 read it, the token runs in fp32 as above (the
// read-out uses the new state as computed), and pass 2 rounds the new state
// to nearest-even bf16 as it stores it.
#include <atomic>

#include "kda_internal.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kHeadDim / kWarps;           // 16
template <bool BF16S>
constexpr int kStateBytes = kHeadDim * kHeadDim * (BF16S ? 2 : 4);   // 32768 or 65536

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// ln(1 + e^x) without overflow.
__device__ __forceinline__ float softplusf_(float x) {
    return x > 0.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

// Four consecutive state elements of row-major row `i`, columns [4 l, 4 l + 4).
template <bool BF16S>
__device__ __forceinline__ float4 load4(const uint8_t* sS, int i, int l) {
    if constexpr (BF16S) {
        const uint2 w = reinterpret_cast<const uint2*>(sS + i * kHeadDim * 2)[l];
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    } else {
        return reinterpret_cast<const float4*>(sS + i * kHeadDim * 4)[l];
    }
}

// bf16 pair {lo, hi} rounded to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <bool BF16S>
__device__ __forceinline__ void store4(uint8_t* sS, int i, int l, float4 t) {
    if constexpr (BF16S) {
        reinterpret_cast<uint2*>(sS + i * kHeadDim * 2)[l] = make_uint2(pack_bf16x2(t.x, t.y), pack_bf16x2(t.z, t.w));
    } else {
        reinterpret_cast<float4*>(sS + i * kHeadDim * 4)[l] = t;
    }
}

// Resident CTAs per SM: 3 for the fp32 state (3 x 75 KiB of shared memory);
// 5 for the bf16 state (43 KiB each), which keeps as many state bytes in
// flight per SM as the fp32 kernel does with 3 (measured on the 256 x 64
// workload: 0.274 ms per call at 3, 0.218 at 4, 0.207 at 5; at 5 the 48
// registers leave an 8-byte spill).
template <bool BF16S>
__global__ void __launch_bounds__(kThreads, BF16S ? 5 : 3)
kda_decode_kernel(const LayerParams p, const DecodeIO io, int* err) {
    constexpr int D = kHeadDim;
    constexpr int kBytes = kStateBytes<BF16S>;
    extern __shared__ __align__(128) uint8_t sS[];        // the 128 x 128 state
    __shared__ float s_q[D], s_k[D], s_v[D], s_a[D];
    __shared__ __align__(16) float s_red_u[kWarps][D];
    __shared__ __align__(16) float s_red_p[kWarps][D];
    __shared__ __align__(16) float s_delta[D];
    __shared__ float s_scal[4];
    __shared__ float s_ms[4];
    __shared__ __align__(8) uint64_t s_bar;

    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    uint8_t* Sg = BF16S ? reinterpret_cast<uint8_t*>(io.S16 + (size_t)bh * D * D)
                        : reinterpret_cast<uint8_t*>(io.S + (size_t)bh * D * D);

    // 1. One bulk copy brings the whole state in.
    if (tid == 0) {
        ptx::mbar_init(&s_bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        ptx::mbar_arrive_expect_tx(&s_bar, kBytes);
        ptx::bulk_g2s(sS, Sg, kBytes, &s_bar);
    }

    // Launched after the low-rank front-end (programmatic dependent launch),
    // the state load above is already in flight while the front-end
    // finishes; z and beta_logit are its results, read below.
    ptx::griddep_wait();

    // 2. While it is in flight: conv4 + SiLU on the 3*d channels of q, k, v
    //    and the per-channel decay a = exp(gk), gk = -exp(A_log) softplus(z +
    //    dt_bias).  The shifted window is held in registers and written back
    //    only once the state load is known to have landed (step 5).
    const size_t HD = (size_t)p.H * D;
    const size_t HD3 = 3 * HD;
    float* win = io.conv_state + (size_t)b * 3 * HD3;
    float wnew[2][3];          // (m2, m1, x_t) of this thread's conv channels
    size_t wgc[2] = {0, 0};
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int ch = tid + it * kThreads;
        if (ch < 3 * D) {
            const int tensor = ch >> 7;
            const int c = ch & (D - 1);
            const size_t gc = (size_t)tensor * HD + (size_t)h * D + c;
            const float* x = tensor == 0 ? io.q : (tensor == 1 ? io.k : io.v);
            const float xt = x[(size_t)bh * D + c];
            const float4 w = *reinterpret_cast<const float4*>(p.conv_w + gc * 4);
            const float m3 = win[gc];
            const float m2 = win[HD3 + gc];
            const float m1 = win[2 * HD3 + gc];
            const float pre = fmaf(w.w, xt, fmaf(w.z, m1, fmaf(w.y, m2, w.x * m3)));
            wgc[it] = gc;
            wnew[it][0] = m2; wnew[it][1] = m1; wnew[it][2] = xt;
            (tensor == 0 ? s_q : (tensor == 1 ? s_k : s_v))[c] = pre / (1.0f + expf(-pre));
        } else {
            const int c = ch - 3 * D;
            const float x = io.z[(size_t)bh * D + c] + p.dt_bias[h * D + c];
            s_a[c] = expf(-expf(p.A_log[h * D + c]) * softplusf_(x));
        }
    }
    __syncthreads();

    // 3. |q|^2, |k|^2, q.k (warps 0..2) and beta (warp 3).
    if (warp < 3) {
        const float* xa = warp == 1 ? s_k : s_q;
        const float* xb = warp == 0 ? s_q : s_k;
        float acc = 0.0f;
#pragma unroll
        for (int j = lane; j < D; j += 32) acc = fmaf(xa[j], xb[j], acc);
        acc = warp_sum(acc);
        if (lane == 0) s_scal[warp] = acc;
    } else if (tid == 96) {
        s_scal[3] = sigmoidf_(io.beta_logit[bh]);
    }
    __syncthreads();
    const float rq = 1.0f / sqrtf(s_scal[0] + p.l2_eps);
    const float rk = 1.0f / sqrtf(s_scal[1] + p.l2_eps);
    const float qk = s_scal[2] * rq * rk;
    const float beta = s_scal[3];

    // Every thread waits (bounded) for the state load; a thread that gives up
    // records the error bit.  Whether the whole CTA saw the load land is
    // decided at the next barrier (all_ok).
    const bool ok = ptx::mbar_wait(&s_bar, 0, err, ptx::kErrDecodeLoadWait);

    // 4. Pass 1: partial u = S'^T k and p = S'^T q over this warp's rows
    //    (the 1/|k| and 1/|q| scales are applied to the column totals).
    const int row0 = warp * kRowsPerWarp;
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 pr = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int i = row0 + r;
        const float ai = s_a[i], ki = s_k[i] * ai, qi = s_q[i] * ai;
        const float4 x = load4<BF16S>(sS, i, lane);
        u.x = fmaf(ki, x.x, u.x); u.y = fmaf(ki, x.y, u.y);
        u.z = fmaf(ki, x.z, u.z); u.w = fmaf(ki, x.w, u.w);
        pr.x = fmaf(qi, x.x, pr.x); pr.y = fmaf(qi, x.y, pr.y);
        pr.z = fmaf(qi, x.z, pr.z); pr.w = fmaf(qi, x.w, pr.w);
    }
    reinterpret_cast<float4*>(s_red_u[warp])[lane] = u;
    reinterpret_cast<float4*>(s_red_p[warp])[lane] = pr;
    const bool all_ok = __syncthreads_and(ok) != 0;
    if (!all_ok) {
        // Give-up path: nothing of this (sequence, head) is written (window,
        // o, o_pre and S keep their old contents); wait once more, bounded,
        // for the state load so that no copy into this CTA's shared memory is
        // left in flight when it exits.
        if (tid == 0) ptx::mbar_wait_timed(&s_bar, 0);
        return;
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        if (tid + it * kThreads < 3 * D) {
            win[wgc[it]] = wnew[it][0];
            win[HD3 + wgc[it]] = wnew[it][1];
            win[2 * HD3 + wgc[it]] = wnew[it][2];
        }
    }

    // 5. Column totals, delta = beta (v - u), o_pre = p + (q^.k^) delta.
    float opre = 0.0f;
    if (tid < D) {
        const int j = tid;
        float uj = 0.0f, pj = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) { uj += s_red_u[w][j]; pj += s_red_p[w][j]; }
        uj *= rk;
        pj *= rq;
        const float delta = beta * (s_v[j] - uj);
        opre = fmaf(qk, delta, pj);
        s_delta[j] = delta * rk;  // k^_i delta_j = k_i (rk delta_j)
        if (io.o_pre) io.o_pre[(size_t)bh * D + j] = opre;
        const float ss = warp_sum(opre * opre);
        if (lane == 0) s_ms[warp] = ss;
    }
    __syncthreads();

    // 6. Pass 2: S_new = Diag(a) S + k^ delta^T in shared memory, then one
    //    bulk store back.
    const float4 dl = reinterpret_cast<const float4*>(s_delta)[lane];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int i = row0 + r;
        const float ai = s_a[i], ki = s_k[i];
        float4 t = load4<BF16S>(sS, i, lane);
        t.x = fmaf(ki, dl.x, t.x * ai); t.y = fmaf(ki, dl.y, t.y * ai);
        t.z = fmaf(ki, dl.z, t.z * ai); t.w = fmaf(ki, dl.w, t.w * ai);
        store4<BF16S>(sS, i, lane, t);
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        ptx::bulk_s2g(Sg, sS, kBytes);
        ptx::bulk_commit();
    }

    // 7. Head RMSNorm, gamma and the sigmoid gate.
    if (tid < D) {
        const int j = tid;
        const float ms = (s_ms[0] + s_ms[1] + s_ms[2] + s_ms[3]) * (1.0f / D);
        const float inv = 1.0f / sqrtf(ms + p.rms_eps);
        const float g = sigmoidf_(io.gate_logit[(size_t)bh * D + j]);
        io.o[(size_t)bh * D + j] = p.gamma[h * D + j] * opre * inv * g;
    }
    // The CTA's shared memory must outlive the bulk store's reads of it.
    if (tid == 0) ptx::bulk_wait_read_all();
}

// Per-device flag: the kernel's attributes are set (the calls are
// idempotent, so two host threads setting them at once is harmless).
std::atomic<bool> g_attr_done[64];

template <bool BF16S>
cudaError_t set_attrs() {
    cudaError_t e = cudaFuncSetAttribute(kda_decode_kernel<BF16S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kStateBytes<BF16S>);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kda_decode_kernel<BF16S>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

}  // namespace

cudaError_t launch_decode(const LayerParams& p, const DecodeIO& io, const DeviceInfo& dev,
                          int* err_word, cudaStream_t stream, bool pdl) {
    const long long grid = (long long)io.B * p.H;
    if (grid <= 0) return cudaSuccess;
    if (dev.device < 0 || dev.device >= 64 || !g_attr_done[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = set_attrs<false>();
        if (e != cudaSuccess) return e;
        e = set_attrs<true>();
        if (e != cudaSuccess) return e;
        if (dev.device >= 0 && dev.device < 64) g_attr_done[dev.device].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = io.S16 ? kStateBytes<true> : kStateBytes<false>;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = io.S16 ? cudaLaunchKernelEx(&cfg, kda_decode_kernel<true>, p, io, err_word)
                                 : cudaLaunchKernelEx(&cfg, kda_decode_kernel<false>, p, io, err_word);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kda
