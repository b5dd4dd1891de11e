// Projections on either side of the token step, on tcgen05 tensor cores.
//
// "Metal (Apple GPU) backend for Kimi K3", table "What runs where (per
// layer)", row "KDA projections (q,k,v,g,o)", and "Kimi K3 Metal Gap
// Analysis", section 2, row "O projection" (W_o[sig(W_g x) * RMSNorm_head(
// S^T q)]): per token,
//
//   [q | k | v | gate_logit] = [W_q; W_k; W_v; W_g] x     (input projections)
//   y                        = W_o o                        (output projection)
//
// with x the layer's hidden input and o the gated, normalised output of the
// token step.  Both are one GEMM C[N][M] = X[N][K] W[M][K]^T over the N
// tokens of a call, bf16 operands with fp32 accumulation:
//
//  * persistent CTAs (one per SM) walk the 128 x Nt output tiles in groups of
//    kGroupM consecutive weight tiles, so that the tiles a wave works on share
//    their weight rows and token rows in L2;
//  * warp 0 streams 64-wide K slices of both operands with TMA (128-byte
//    swizzle) through a ring of 4 stages; warp 1 issues kind::f16 MMAs
//    (M = 128, N = Nt, K = 16, four per slice) into one of two TMEM
//    accumulators and releases each stage with a commit; warps 2-5 read the
//    other accumulator back (TMEM lane = output feature) while the next tile
//    accumulates, and store it token-major, each 128-row tile into the
//    output tensor it belongs to (q, k, v as bf16 or fp32, gate logits and y
//    as fp32): per token, a warp writes 32 consecutive features.
//
// The output projection takes o in fp32; a conversion kernel writes its bf16
// copy into the caller's workspace first (round to nearest even).  When its
// output tiles would leave more than half of the SMs idle (a few tokens: the
// call then streams W_o), K is split in two halves on separate CTAs, each
// adding its fp32 partial tile into y (zeroed by the conversion kernel) with
// red.global.add: with exactly two addends onto zero, (0 + a) + b and
// (0 + b) + a are the same float, so y does not depend on their order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "kda_internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kMaxStages = 8;
constexpr uint32_t kRingBudget = 192 * 1024;     // shared memory for the ring of stages
constexpr int kKSlice = 64;                      // bf16 elements in one 128-byte swizzled row
constexpr uint32_t kATile = 128 * 128;           // 128 weight rows x 128 bytes
constexpr int kThreads = 192;                    // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kEpiThreads = 128;
constexpr int kGroupM = 16;                      // weight tiles per raster group
constexpr int kMaxSegs = 4;

struct Seg {
    void* ptr;      // [N][len] row-major
    int len;        // features of this output (a multiple of 128)
    int bf16;       // 1: store bf16 (round to nearest even), 0: store fp32
};

struct ProjArgs {
    int M, N, K;            // C[N][M] = X[N][K] W[M][K]^T
    int Nt;                 // token tile: 32, 64, 128 or 256
    int mtiles, ntiles;
    int ksplit;             // K halves per tile: 1, or 2 (fp32 output added into, zero on entry)
    int stages;             // depth of the ring, ring_stages(Nt)
    int nsegs;              // outputs, each `len` consecutive features of M
    Seg seg[kMaxSegs];
};

struct ProjMaps {
    CUtensorMap w;   // (K, M), boxes of (64, 128)
    CUtensorMap x;   // (K, N), boxes of (64, Nt)
};

__host__ __device__ constexpr uint32_t stage_bytes(int Nt) { return kATile + (uint32_t)Nt * 128; }
// Ring depth: as many stages as 192 KiB holds, at most 8 (8 at 32 and 64
// tokens, 6 at 128, 4 at 256).  A token-light call streams its weights at a
// rate set by the bytes it keeps in flight per SM, so small tiles get more
// stages.
constexpr int ring_stages(int Nt) {
    return (int)(kRingBudget / stage_bytes(Nt)) < kMaxStages ? (int)(kRingBudget / stage_bytes(Nt)) : kMaxStages;
}
constexpr uint32_t proj_smem_bytes(int Nt) { return ring_stages(Nt) * stage_bytes(Nt) + 1024; }
constexpr uint32_t max_u32(uint32_t a, uint32_t b) { return a > b ? a : b; }
constexpr uint32_t kMaxSmem = max_u32(max_u32(proj_smem_bytes(32), proj_smem_bytes(64)),
                                      max_u32(proj_smem_bytes(128), proj_smem_bytes(256)));

__device__ __forceinline__ void red_add(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, int* dead, int* err) {
    if (*(volatile int*)dead) return false;
    if (ptx::mbar_wait_timed(bar, parity, dead)) return true;
    *(volatile int*)dead = 1;
    atomicOr(err, ptx::kErrProjWait);
    return false;
}

// Tile t -> (weight tile, token tile): groups of kGroupM weight tiles, the
// token tiles walked inside a group.
__device__ __forceinline__ void raster(const ProjArgs& g, int t, int& mt, int& nt) {
    const int per = kGroupM * g.ntiles;
    const int grp = t / per;
    const int first = grp * kGroupM;
    const int size = min(kGroupM, g.mtiles - first);
    const int in = t - grp * per;
    mt = first + in % size;
    nt = in / size;
}

__global__ void __launch_bounds__(kThreads, 1)
kda_proj_gemm_kernel(const ProjArgs g, int* err, const __grid_constant__ ProjMaps maps) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbytes = stage_bytes(g.Nt);
    const int S = g.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S * sbytes);         // slice landed
    uint64_t* empty = full + kMaxStages;                                   // slice consumed
    uint64_t* accf = empty + kMaxStages;                                   // [2] accumulator complete
    uint64_t* acce = accf + 2;                                             // [2] accumulator read back
    uint64_t* drain = acce + 2;                                            // give-up path
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain + 1);
    int* s_dead = reinterpret_cast<int*>(s_tmem + 1);
    int* s_issued = s_dead + 1;

    // Work unit u = (tile u / ksplit, K range u % ksplit): K slices [k0, k1).
    const int units = g.mtiles * g.ntiles * g.ksplit;
    const int nk = (g.K + kKSlice - 1) / kKSlice;
    auto krange = [&](int u, int& k0, int& k1) {
        const int ks = u % g.ksplit;
        k0 = ks * nk / g.ksplit;
        k1 = (ks + 1) * nk / g.ksplit;
    };
    const uint32_t ncols = 2u * (uint32_t)g.Nt;   // two accumulators

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&accf[b], 1);
            ptx::mbar_init(&acce[b], kEpiThreads);
        }
        ptx::mbar_init(drain, 1);
        ptx::fence_mbar_init();
        *s_dead = 0;
        *s_issued = 0;
    }
    if (warp == 0) tc::alloc(s_tmem, ncols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *s_tmem;
    // Output projection (programmatic dependent launch): the conversion
    // kernel before has written x and zeroed y once this returns.
    ptx::griddep_wait();

    if (tid == 0) {
        // TMA producer: slices of every tile of this CTA, in order; slice it
        // goes to stage s = it % S, rp = parity of it / S.
        int it = 0, s = 0;
        uint32_t rp = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x) {
            int mt, nt, k0, k1;
            raster(g, u / g.ksplit, mt, nt);
            krange(u, k0, k1);
            for (int i = k0; i < k1; ++i, ++it) {
                if (it >= S && !pwait(&empty[s], rp ^ 1u, s_dead, err)) goto done_p;
                uint8_t* st = sm + s * sbytes;
                ptx::mbar_arrive_expect_tx(&full[s], sbytes);
                ptx::tma_load_2d(st, &maps.w, i * kKSlice, mt * 128, &full[s]);
                ptx::tma_load_2d(st + kATile, &maps.x, i * kKSlice, nt * g.Nt, &full[s]);
                *s_issued = it + 1;
                if (++s == S) { s = 0; rp ^= 1u; }
            }
        }
    done_p:;
    } else if (tid == 32) {
        // MMA issuer: tile j accumulates into TMEM columns [(j & 1) Nt, + Nt)
        // once the epilogue has read that accumulator's previous tile.
        const uint32_t id = tc::idesc_bf16(128, g.Nt);
        int j = 0, s = 0;
        uint32_t rp = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
            const int b = j & 1;
            if (j >= 2 && !pwait(&acce[b], (uint32_t)(((j >> 1) - 1) & 1), s_dead, err)) break;
            tc::fence_after();
            const uint32_t d = tm + (uint32_t)(b * g.Nt);
            int k0, k1;
            krange(u, k0, k1);
            bool ok = true;
            for (int i = k0; i < k1; ++i) {
                if (!pwait(&full[s], rp, s_dead, err)) { ok = false; break; }
                tc::fence_after();
                const uint64_t da = tc::desc_sw128(ptx::smem_u32(sm + s * sbytes));
                const uint64_t db = tc::desc_add(da, kATile);
#pragma unroll
                for (int kin = 0; kin < 4; ++kin)
                    tc::mma_ss_bf16(d, tc::desc_add(da, kin * 32), tc::desc_add(db, kin * 32), id,
                                    (i > k0 || kin > 0) ? 1u : 0u);
                tc::commit(&empty[s]);
                if (++s == S) { s = 0; rp ^= 1u; }
            }
            tc::commit(&accf[b]);
            if (!ok) break;
        }
        tc::commit(drain);   // completes once every MMA this thread issued has completed
    } else if (warp >= 2) {
        // Epilogue: TMEM lane r = output feature mt * 128 + r, column = token.
        const int r = 32 * (warp & 3) + lane;
        int j = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
            const int b = j & 1;
            if (!pwait(&accf[b], (uint32_t)((j >> 1) & 1), s_dead, err)) break;
            tc::fence_after();
            const int t = u / g.ksplit;
            int mt, nt;
            raster(g, t, mt, nt);
            const int n0 = nt * g.Nt;
            if (g.ksplit > 1) {
                // Split K: this half's fp32 partial tile added into the
                // (single, fp32) output, token-major (a warp adds 32
                // consecutive features per token).
                float* out = static_cast<float*>(g.seg[0].ptr) + mt * 128 + r;
                for (int c0 = 0; c0 < g.Nt; c0 += 32) {
                    uint32_t v[32];
                    tc::ld32(tc::taddr(tm, warp, b * g.Nt + c0), v);
                    tc::wait_ld();
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int n = n0 + c0 + q;
                        if (n < g.N) red_add(out + (size_t)n * g.M, __uint_as_float(v[q]));
                    }
                }
                tc::fence_before();
                ptx::mbar_arrive(&acce[b]);
                continue;
            }
            int off = mt * 128 + r;   // feature index, then the offset inside its output
            Seg sg = g.seg[0];
#pragma unroll
            for (int i = 1; i < kMaxSegs; ++i)
                if (i < g.nsegs && off >= sg.len) {
                    off -= sg.len;
                    sg = g.seg[i];
                }
            for (int c0 = 0; c0 < g.Nt; c0 += 32) {
                uint32_t v[32];
                tc::ld32(tc::taddr(tm, warp, b * g.Nt + c0), v);
                tc::wait_ld();
                if (sg.bf16) {
                    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.ptr) + off;
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int n = n0 + c0 + q;
                        if (n < g.N) out[(size_t)n * sg.len] = __float2bfloat16_rn(__uint_as_float(v[q]));
                    }
                } else {
                    float* out = static_cast<float*>(sg.ptr) + off;
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int n = n0 + c0 + q;
                        if (n < g.N) out[(size_t)n * sg.len] = __uint_as_float(v[q]);
                    }
                }
            }
            tc::fence_before();
            ptx::mbar_arrive(&acce[b]);
        }
    }

    tc::fence_before();
    const bool dead = __syncthreads_or(*(volatile int*)s_dead) != 0;
    if (dead) {
        // Give-up path: the MMAs and the copies this CTA issued complete
        // (bounded waits) before its TMEM and shared memory are released.
        if (tid == 32) ptx::mbar_wait_timed(drain, 0);
        if (tid == 0) {
            const int issued = *s_issued;
            for (int s = 0; s < S && s < issued; ++s) {
                const int uses = (issued - s + S - 1) / S;
                ptx::mbar_wait_timed(&full[s], (uint32_t)((uses - 1) & 1));
            }
        }
    }
    __syncthreads();
    if (warp == 0) tc::dealloc(tm, ncols);
}

// o (fp32) -> bf16, round to nearest even; n is a multiple of 4.
// With split K it also zeroes y (nz4 float4s), which the GEMM then adds into.
__global__ void kda_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out, size_t n4,
                                   float4* __restrict__ zero, size_t nz4) {
    ptx::griddep_launch_dependents();   // the GEMM may set up meanwhile
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nz4; i += (size_t)gridDim.x * blockDim.x)
        zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 a = in[i];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
        out[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
}

std::atomic<bool> g_attr_done[64];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Row-major bf16 [rows][K] seen as 2-D (K, rows), boxes of (64, box_rows),
// 128-byte swizzle; rows and columns past the end read as zeros.
bool make_map_bf16(CUtensorMap* m, const void* base, int K, int rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kKSlice, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int token_tile(int N) {
    int t = 32;
    while (t < N && t < 256) t <<= 1;
    return t;
}

// K halves per output tile: 2 when the tiles would leave more than half of
// the SMs idle and K spans at least 16 slices of 64, else 1.
int ksplit_for(int M, int N, int K, int sm_count) {
    const int Nt = token_tile(N);
    const long long tiles = (long long)(M / 128) * ((N + Nt - 1) / Nt);
    const int nk = (K + kKSlice - 1) / kKSlice;
    return (tiles > 0 && 2 * tiles <= sm_count && nk >= 16) ? 2 : 1;
}

cudaError_t run_proj(const CUtensorMap& wmap, int M, const void* x, int N, int K, const Seg* segs, int nsegs,
                     int ksplit, const DeviceInfo& dev, int* err_word, cudaStream_t stream, bool pdl) {
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!g_attr_done[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kda_proj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kMaxSmem);
        if (e != cudaSuccess) return e;
        g_attr_done[dev.device].store(true, std::memory_order_release);
    }
    ProjArgs g{};
    g.M = M;
    g.N = N;
    g.K = K;
    g.Nt = token_tile(N);
    g.mtiles = M / 128;
    g.ntiles = (N + g.Nt - 1) / g.Nt;
    g.ksplit = ksplit;
    g.stages = ring_stages(g.Nt);
    g.nsegs = nsegs;
    for (int i = 0; i < nsegs; ++i) g.seg[i] = segs[i];
    ProjMaps maps{};
    maps.w = wmap;
    if (!make_map_bf16(&maps.x, x, K, N, g.Nt)) return cudaErrorInvalidValue;
    const int units = g.mtiles * g.ntiles * g.ksplit;
    const int grid = units < dev.sm_count ? units : dev.sm_count;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = proj_smem_bytes(g.Nt);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kda_proj_gemm_kernel, g, err_word, maps);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool proj_prepare(const LayerParams& p, Projections& pr) {
    const int HD = p.H * kHeadDim;
    pr.maps_ready = make_map_bf16(&pr.map_qkvg, pr.W_qkvg, pr.hidden, 4 * HD, 128) &&
                    make_map_bf16(&pr.map_o, pr.W_o, HD, pr.hidden, 128);
    return pr.maps_ready;
}

cudaError_t launch_project_qkvg(const LayerParams& p, const Projections& pr, int N, const void* x, void* q,
                                void* k, void* v, float* gate_logit, bool qkv_f32, const DeviceInfo& dev,
                                int* err_word, cudaStream_t stream) {
    if (N <= 0) return cudaSuccess;
    if (!pr.maps_ready) return cudaErrorInvalidValue;
    const int HD = p.H * kHeadDim;
    const int b = qkv_f32 ? 0 : 1;
    const Seg segs[4] = {{q, HD, b}, {k, HD, b}, {v, HD, b}, {gate_logit, HD, 0}};
    return run_proj(pr.map_qkvg, 4 * HD, x, N, pr.hidden, segs, 4, 1, dev, err_word, stream, false);
}

int project_o_ksplit(int hidden, int N, int HD, int sm_count) { return ksplit_for(hidden, N, HD, sm_count); }

size_t project_o_workspace_bytes(const LayerParams& p, int N) {
    return N <= 0 ? 0 : (size_t)N * p.H * kHeadDim * 2;
}

cudaError_t launch_project_o(const LayerParams& p, const Projections& pr, int N, const float* o, float* y,
                             void* workspace, const DeviceInfo& dev, int* err_word, cudaStream_t stream) {
    if (N <= 0) return cudaSuccess;
    if (!pr.maps_ready) return cudaErrorInvalidValue;
    const int HD = p.H * kHeadDim;
    const int ksplit = ksplit_for(pr.hidden, N, HD, dev.sm_count);
    const size_t n4 = (size_t)N * HD / 4;
    const size_t nz4 = ksplit > 1 ? (size_t)N * pr.hidden / 4 : 0;
    const size_t work = n4 > nz4 ? n4 : nz4;
    const size_t want = (work + 255) / 256, cap = (size_t)dev.sm_count * 16;
    kda_to_bf16_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(o), static_cast<uint2*>(workspace), n4, reinterpret_cast<float4*>(y), nz4);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const Seg segs[1] = {{y, pr.hidden, 0}};
    return run_proj(pr.map_o, pr.hidden, workspace, N, HD, segs, 1, ksplit, dev, err_word, stream, true);
}

}  // namespace kda
