// Prefill, first correct form: one CTA per (sequence, head) walks the T
// tokens in order with the 128x128 fp32 state held in registers for the
// whole sequence (read once, written once).  Same per-token arithmetic as
// the decode kernel ("Kimi K3 Metal Gap Analysis", section 2 "KDA
// Attention", rows "Conv4 + SiLU" to "O projection").
#include <cuda_bf16.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kHeadDim / kWarps;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) {
    return x > 0.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__global__ void __launch_bounds__(kThreads, 1)
kda_prefill_seq_kernel(const LayerParams p, const PrefillIO io) {
    constexpr int D = kHeadDim;
    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, T = io.T;

    __shared__ float s_q[D], s_k[D], s_v[D], s_a[D];
    __shared__ __align__(16) float s_red_u[kWarps][D];
    __shared__ __align__(16) float s_red_p[kWarps][D];
    __shared__ __align__(16) float s_delta[D];
    __shared__ float s_scal[4];
    __shared__ float s_ms[4];

    float* Sg = io.S + (size_t)bh * D * D;
    const int row0 = warp * kRowsPerWarp;
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
        s[r] = reinterpret_cast<const float4*>(Sg + (size_t)(row0 + r) * D)[lane];

    // Conv windows of the (up to two) channels this thread owns, in registers.
    const size_t HD = (size_t)H * D, HD3 = 3 * HD;
    float* win = io.conv_state + (size_t)b * 3 * HD3;
    float wm[2][3];
    float4 wt[2];
    size_t gch[2];
    int nch = 0;
    for (int ch = tid; ch < 3 * D; ch += kThreads, ++nch) {
        const int tensor = ch >> 7, c = ch & (D - 1);
        gch[nch] = (size_t)tensor * HD + (size_t)h * D + c;
        wt[nch] = *reinterpret_cast<const float4*>(p.conv_w + gch[nch] * 4);
        wm[nch][0] = win[gch[nch]];
        wm[nch][1] = win[HD3 + gch[nch]];
        wm[nch][2] = win[2 * HD3 + gch[nch]];
    }
    float A_exp = 0.f, dtb = 0.f;
    if (tid >= kThreads - D) {
        const int c = tid - (kThreads - D);
        A_exp = expf(p.A_log[h * D + c]);
        dtb = p.dt_bias[h * D + c];
    }
    const float gam = tid < D ? p.gamma[h * D + tid] : 0.f;

    for (int t = 0; t < T; ++t) {
        const size_t row = (((size_t)b * T + t) * H + h) * D;
        for (int n = 0; n < nch; ++n) {
            const int ch = tid + n * kThreads;
            const int tensor = ch >> 7, c = ch & (D - 1);
            const uint16_t* x = tensor == 0 ? io.q : (tensor == 1 ? io.k : io.v);
            const float xt = bf16_to_f32(x[row + c]);
            const float4 w = wt[n];
            const float pre = fmaf(w.w, xt, fmaf(w.z, wm[n][2], fmaf(w.y, wm[n][1], w.x * wm[n][0])));
            wm[n][0] = wm[n][1];
            wm[n][1] = wm[n][2];
            wm[n][2] = xt;
            (tensor == 0 ? s_q : (tensor == 1 ? s_k : s_v))[c] = pre / (1.0f + expf(-pre));
        }
        if (tid >= kThreads - D) {
            const int c = tid - (kThreads - D);
            const float gk = -A_exp * softplusf_(io.z[row + c] + dtb);
            s_a[c] = expf(gk);
        }
        __syncthreads();
        if (warp < 3) {
            const float* xa = warp == 1 ? s_k : s_q;
            const float* xb = warp == 0 ? s_q : s_k;
            float acc = 0.0f;
#pragma unroll
            for (int j = lane; j < D; j += 32) acc = fmaf(xa[j], xb[j], acc);
            acc = warp_sum(acc);
            if (lane == 0) s_scal[warp] = acc;
        } else if (tid == 96) {
            s_scal[3] = sigmoidf_(io.beta_logit[((size_t)b * T + t) * H + h]);
        }
        __syncthreads();
        const float rq = 1.0f / sqrtf(s_scal[0] + p.l2_eps);
        const float rk = 1.0f / sqrtf(s_scal[1] + p.l2_eps);
        const float qk = s_scal[2] * rq * rk;
        const float beta = s_scal[3];

        float4 u = make_float4(0.f, 0.f, 0.f, 0.f), pr = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int i = row0 + r;
            const float ai = s_a[i], ki = s_k[i], qi = s_q[i];
            s[r].x *= ai; s[r].y *= ai; s[r].z *= ai; s[r].w *= ai;
            u.x = fmaf(ki, s[r].x, u.x); u.y = fmaf(ki, s[r].y, u.y);
            u.z = fmaf(ki, s[r].z, u.z); u.w = fmaf(ki, s[r].w, u.w);
            pr.x = fmaf(qi, s[r].x, pr.x); pr.y = fmaf(qi, s[r].y, pr.y);
            pr.z = fmaf(qi, s[r].z, pr.z); pr.w = fmaf(qi, s[r].w, pr.w);
        }
        reinterpret_cast<float4*>(s_red_u[warp])[lane] = u;
        reinterpret_cast<float4*>(s_red_p[warp])[lane] = pr;
        __syncthreads();
        float opre = 0.f;
        if (tid < D) {
            const int j = tid;
            float uj = 0.f, pj = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) { uj += s_red_u[w][j]; pj += s_red_p[w][j]; }
            uj *= rk;
            pj *= rq;
            const float delta = beta * (s_v[j] - uj);
            opre = fmaf(qk, delta, pj);
            s_delta[j] = delta * rk;
            const float ss = warp_sum(opre * opre);
            if (lane == 0) s_ms[warp] = ss;
        }
        __syncthreads();
        const float4 dl = reinterpret_cast<const float4*>(s_delta)[lane];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float ki = s_k[row0 + r];
            s[r].x = fmaf(ki, dl.x, s[r].x); s[r].y = fmaf(ki, dl.y, s[r].y);
            s[r].z = fmaf(ki, dl.z, s[r].z); s[r].w = fmaf(ki, dl.w, s[r].w);
        }
        if (tid < D) {
            const float ms = (s_ms[0] + s_ms[1] + s_ms[2] + s_ms[3]) * (1.0f / D);
            const float inv = 1.0f / sqrtf(ms + p.rms_eps);
            io.o[row + tid] = gam * opre * inv * sigmoidf_(io.gate_logit[row + tid]);
        }
        __syncthreads();  // s_q/s_k/s_v/s_a are rewritten by the next token
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
        reinterpret_cast<float4*>(Sg + (size_t)(row0 + r) * D)[lane] = s[r];
    for (int n = 0; n < nch; ++n) {
        win[gch[n]] = wm[n][0];
        win[HD3 + gch[n]] = wm[n][1];
        win[2 * HD3 + gch[n]] = wm[n][2];
    }
}

}  // namespace

size_t prefill_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_prefill(const LayerParams& p, const PrefillIO& io, const DeviceInfo&, int*,
                           cudaStream_t stream) {
    const long long grid = (long long)io.B * p.H;
    if (grid <= 0 || io.T <= 0) return cudaSuccess;
    kda_prefill_seq_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(p, io);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kda
