// Low-rank front-end of the decay and beta inputs, on tcgen05 tensor cores.
//
// "Metal (Apple GPU) backend for Kimi K3", table "What runs where (per
// layer)", row "KDA low-rank (fa,fb,bp)", and "Kimi K3 Metal Gap Analysis",
// section 2, row "Decay compute" (z = W_fb W_fa x): per token with hidden
// input x,
//
//   u          = W_fa x     (rank)
//   z          = W_fb u     (H * d: the decay input of every head)
//   beta_logit = W_bp x     (H)
//
// These are dense contractions shared by every head of a token (u) and by
// every token (the weights), so they run as GEMMs over all N tokens of a call
// before the per-(sequence, head) kernels, not inside them:
//
//   GEMM A  [u | beta_logit]^T = [W_fa ; W_bp] x^T, split over K (hidden) so
//           that a decode batch of 64..256 tokens still spreads over the SMs;
//           partial sums go to the workspace;
//   reduce  the partial sums in a fixed order (deterministic) into u and
//           beta_logit;
//   GEMM C  z^T = W_fb u^T.
//
// One GEMM kernel serves both: C[n][m] = sum_k A[m][k] B[n][k] with A the
// weights (row-major [rows][K], i.e. K-major) and B the activations
// (row-major [N][K], K-major too), fp32 accumulation in TMEM.  The products
// keep fp32 accuracy with three tf32 MMAs per product (the split of each
// operand a = hi + lo, hi its tf32 truncation): hi*hi + hi*lo + lo*hi, whose
// dropped lo*lo term and tf32 rounding of lo are below 2^-20 of the product.
// (A single tf32 product would leave z about 5e-4 off at K = 7168, and z
// reaches the state through e^gk at every token.)  The MMA itself reads an
// fp32 operand as its tf32 truncation, so the TMA-landed tile serves as hi;
// two warps write lo = a - hi beside it.
//
// A CTA owns a 128-row tile of A, an N tile of 32 to 256 tokens and one K
// split; one thread (warp 0) streams 32-wide K slices of both operands with
// TMA (128-byte swizzle) through a ring of stages, warps 2-5 form the lo
// parts of each landed slice, one thread (warp 1) issues the kind::tf32 MMAs
// (M = 128, N = the tile, 3 x 4 per slice) and releases the stage with a
// commit.  Warps 2-5 then read the accumulator back (TMEM lane = output
// row), transpose it through shared memory and store it token-major with
// 16-byte stores, a row of 128 outputs (512 contiguous bytes) per token.
// The weights' tensor maps are encoded once, when the weights are bound.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "kda_internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kMaxStages = 4;
constexpr uint32_t kStageBudget = 200 * 1024;    // shared memory for the ring
constexpr int kKStep = 32;                       // fp32 elements in one 128-byte swizzled row
constexpr uint32_t kATileBytes = 128 * 128;      // 128 rows x 128 bytes
constexpr int kThreads = 192;                    // warp 0 TMA, warp 1 MMA, warps 2-5 split + epilogue
constexpr int kSplitThreads = 128;

struct GemmMaps {
    CUtensorMap a0, a1;   // weights, (K, rows) with boxes of (32, 128)
    CUtensorMap b;        // activations, (K, N) with boxes of (32, Nt)
};

struct GemmArgs {
    int tiles0;     // 128-row tiles taken from the first weight matrix (the rest from the second)
    int N, K;
    int Nt;         // token tile: 32, 64, 128 or 256
    int kslice;     // K elements per split, a multiple of 32
    int stages;     // depth of the ring
    int ldo;        // row stride of the output: 128 x (number of 128-row tiles)
    float* out;     // [splits][N][ldo]; tile t owns columns [128 t, 128 t + 128)
};

// A stage: A hi, B hi (TMA), then A lo, B lo (split warps); each part a
// multiple of 1024 bytes, so every operand starts on a swizzle atom.
__host__ __device__ constexpr uint32_t half_bytes(int Nt) { return kATileBytes + (uint32_t)Nt * 128; }
__host__ __device__ constexpr uint32_t stage_bytes(int Nt) { return 2 * half_bytes(Nt); }
constexpr int ring_stages(int Nt) {
    return (int)(kStageBudget / stage_bytes(Nt)) < kMaxStages ? (int)(kStageBudget / stage_bytes(Nt)) : kMaxStages;
}
constexpr uint32_t gemm_smem_bytes(int Nt) { return ring_stages(Nt) * stage_bytes(Nt) + 1024; }

// Bounded wait shared by the roles of the GEMM CTA: gives up after the wall
// time limit (or at once when another thread already gave up), marks the CTA
// dead and records the error bit.
__device__ __forceinline__ bool gwait(uint64_t* bar, uint32_t parity, int* dead, int* err) {
    if (*(volatile int*)dead) return false;
    if (ptx::mbar_wait_timed(bar, parity, dead)) return true;
    *(volatile int*)dead = 1;
    atomicOr(err, ptx::kErrLowrankWait);
    return false;
}

__device__ __forceinline__ uint32_t lo_part(uint32_t a) {
    return __float_as_uint(__uint_as_float(a) - __uint_as_float(a & 0xffffe000u));
}

__global__ void __launch_bounds__(kThreads, 1)
kda_lowrank_gemm_kernel(const GemmArgs g, int* err, const __grid_constant__ GemmMaps maps) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = g.stages;
    const uint32_t hbytes = half_bytes(g.Nt), sbytes = stage_bytes(g.Nt);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S * sbytes);   // slice landed (hi parts)
    uint64_t* split = full + kMaxStages;                             // lo parts written
    uint64_t* empty = split + kMaxStages;                            // slice consumed by the MMAs
    uint64_t* accb = empty + kMaxStages;                             // accumulator complete
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(accb + 1);
    int* s_dead = reinterpret_cast<int*>(s_tmem + 1);
    int* s_issued = s_dead + 1;                                      // slices the producer issued

    // The next kernel of the front-end (or the decode after it) may start its
    // own set-up now; it waits for this one's results itself.
    ptx::griddep_launch_dependents();
    const int mt = blockIdx.x, nt = blockIdx.y, ks = blockIdx.z;
    const bool second = mt >= g.tiles0;
    const int arow = (second ? mt - g.tiles0 : mt) * 128;    // first row of the tile in its matrix
    const int n0 = nt * g.Nt;
    const int k0 = ks * g.kslice;
    const int k1 = min(g.K, k0 + g.kslice);
    const int nk = (k1 - k0 + kKStep - 1) / kKStep;          // >= 1: the host makes no empty split
    const uint32_t ncols = (uint32_t)g.Nt;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&split[s], kSplitThreads);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(accb, 1);
        ptx::fence_mbar_init();
        *s_dead = 0;
        *s_issued = 0;
    }
    if (warp == 0) tc::alloc(s_tmem, ncols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *s_tmem;
    const CUtensorMap* amap = second ? &maps.a1 : &maps.a0;

    if (tid == 0) {
        // TMA producer: slice i goes to stage i % S once the MMAs of slice
        // i - S have released it.  The B operand of GEMM C is the reduction's
        // output: the kernel before must have completed.
        ptx::griddep_wait();
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (i >= S && !gwait(&empty[s], (uint32_t)((i / S - 1) & 1), s_dead, err)) break;
            uint8_t* st = sm + s * sbytes;
            ptx::mbar_arrive_expect_tx(&full[s], hbytes);
            ptx::tma_load_2d(st, amap, k0 + i * kKStep, arow, &full[s]);
            ptx::tma_load_2d(st + kATileBytes, &maps.b, k0 + i * kKStep, n0, &full[s]);
            *s_issued = i + 1;
        }
    } else if (tid == 32) {
        // MMA issuer: per 32-wide slice, for each K = 8 step, hi*hi, hi*lo and
        // lo*hi; then release the stage.
        const uint32_t id = tc::idesc_tf32(128, g.Nt);
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (!gwait(&split[s], (uint32_t)((i / S) & 1), s_dead, err)) break;
            tc::fence_after();
            const uint32_t ah = ptx::smem_u32(sm + s * sbytes), bh = ah + kATileBytes;
            const uint32_t al = ah + hbytes, bl = al + kATileBytes;
#pragma unroll
            for (int kin = 0; kin < 4; ++kin) {
                tc::mma_ss(tm, tc::desc_sw128(ah + kin * 32), tc::desc_sw128(bh + kin * 32), id,
                           (i | kin) != 0 ? 1u : 0u);
                tc::mma_ss(tm, tc::desc_sw128(ah + kin * 32), tc::desc_sw128(bl + kin * 32), id, 1u);
                tc::mma_ss(tm, tc::desc_sw128(al + kin * 32), tc::desc_sw128(bh + kin * 32), id, 1u);
            }
            tc::commit(&empty[s]);
        }
        tc::commit(accb);   // completes once every MMA this thread issued has completed
    } else if (warp >= 2) {
        // Split warps: lo = a - trunc_tf32(a) for every element of the slice
        // (same byte offsets, so the swizzle carries over), made visible to
        // the tensor cores, then one arrival each on the stage's split
        // barrier.  Four 16-byte words per thread are loaded before any of
        // them is stored.
        const uint32_t t = (uint32_t)(tid - 64);
        const uint32_t n4 = hbytes / 16;
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (!gwait(&full[s], (uint32_t)((i / S) & 1), s_dead, err)) break;
            const uint4* hi = reinterpret_cast<const uint4*>(sm + s * sbytes);
            uint4* lo = reinterpret_cast<uint4*>(sm + s * sbytes + hbytes);
            for (uint32_t j = t; j < n4; j += 4 * kSplitThreads) {
                uint4 a[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j + q * kSplitThreads < n4) a[q] = hi[j + q * kSplitThreads];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j + q * kSplitThreads < n4)
                        lo[j + q * kSplitThreads] =
                            make_uint4(lo_part(a[q].x), lo_part(a[q].y), lo_part(a[q].z), lo_part(a[q].w));
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&split[s]);
        }
    }

    if (warp >= 2) gwait(accb, 0, s_dead, err);
    tc::fence_before();
    const bool dead = __syncthreads_or(*(volatile int*)s_dead) != 0;
    tc::fence_after();
    if (!dead) {
        // Epilogue (warps 2-5; warp w reads TMEM lanes 32 (w % 4) ..): the
        // tile as [Nt][128] fp32 in the ring (every slice has been consumed),
        // then 512-byte rows to the output, one per token.
        float* T = reinterpret_cast<float*>(sm);
        if (warp >= 2) {
            const int r = 32 * (warp & 3) + lane;
            for (int c0 = 0; c0 < g.Nt; c0 += 32) {
                uint32_t v[32];
                tc::ld32(tc::taddr(tm, warp, c0), v);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) T[(c0 + j) * 128 + r] = __uint_as_float(v[j]);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kSplitThreads) : "memory");
            float* out = g.out + ((size_t)ks * g.N + n0) * g.ldo + 128 * mt;
            const int rows = min(g.Nt, g.N - n0);
            for (int idx = tid - 64; idx < rows * 32; idx += kSplitThreads) {
                const int n = idx >> 5, c4 = idx & 31;
                reinterpret_cast<float4*>(out + (size_t)n * g.ldo)[c4] =
                    reinterpret_cast<const float4*>(T + n * 128)[c4];
            }
        }
    } else if (tid == 0) {
        // Give-up path: every slice the producer issued has landed (bounded
        // waits) before the shared memory is released ...
        const int issued = *s_issued;
        for (int s = 0; s < S && s < issued; ++s) {
            const int uses = (issued - s + S - 1) / S;
            ptx::mbar_wait_timed(&full[s], (uint32_t)((uses - 1) & 1));
        }
    } else if (tid == 32) {
        ptx::mbar_wait_timed(accb, 0);   // ... and every MMA has completed before TMEM is freed
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tm, ncols);
}

// Partial sums of GEMM A over the K splits into u [N][M0] and beta_logit
// [N][M1]; partial row n holds tile t's outputs at columns [128 t, 128 t +
// 128) (u tiles first).  A block takes 32 consecutive outputs: warp g sums
// the splits g, g + 8, g + 16, ... of each (coalesced loads, independent of
// one another), and warp 0 adds the eight warp sums in warp order, so the
// order of the additions is fixed (results do not vary from run to run).
constexpr int kReduceWarps = 8;

__global__ void __launch_bounds__(32 * kReduceWarps)
kda_lowrank_reduce_kernel(const float* __restrict__ part, int splits, int N, int ldo, int M0, int M1,
                          int col1, float* __restrict__ u, float* __restrict__ beta_logit) {
    __shared__ float sp[kReduceWarps][32];
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // GEMM A's partial sums
    const size_t M = (size_t)(M0 + M1);
    const size_t total = (size_t)N * M;
    const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
    const size_t i = (size_t)blockIdx.x * 32 + lane;
    size_t n = 0, m = 0, src = 0;
    if (i < total) {
        n = i / M;
        m = i - n * M;
        src = n * ldo + (m < (size_t)M0 ? m : col1 + (m - M0));
    }
    const size_t plane = (size_t)N * ldo;
    float s = 0.0f;
    if (i < total) {
#pragma unroll 4
        for (int k = g; k < splits; k += kReduceWarps) s += part[(size_t)k * plane + src];
    }
    sp[g][lane] = s;
    __syncthreads();
    if (g == 0 && i < total) {
        float t = sp[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceWarps; ++w) t += sp[w][lane];
        if (m < (size_t)M0) u[n * M0 + m] = t;
        else beta_logit[n * M1 + (m - M0)] = t;
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

// Row-major fp32 [rows][K] seen as 2-D (K, rows), boxes of (32, box_rows),
// 128-byte swizzle; rows and columns past the end read as zeros.
bool make_map2d(CUtensorMap* m, const float* base, int K, int rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kKStep, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token tile: a power of two from 32 to 256.
int token_tile(int N) {
    int t = 32;
    while (t < N && t < 256) t <<= 1;
    return t;
}

struct Plan {
    int Nt, ntiles, tiles0, tiles1, kslice, splits, ldo;
};

// Tiling of the output [N][128 x tiles] of [A0; A1] B^T: the K dimension is
// split so that the grid holds about one CTA per SM, each split keeping at
// least four 32-wide slices.
Plan plan_gemm(int M0, int M1, int N, int K, int sm_count) {
    Plan p{};
    p.Nt = token_tile(N);
    p.ntiles = (N + p.Nt - 1) / p.Nt;
    p.tiles0 = (M0 + 127) / 128;
    p.tiles1 = (M1 + 127) / 128;
    p.ldo = 128 * (p.tiles0 + p.tiles1);
    const int ksteps = (K + kKStep - 1) / kKStep;
    const int tiles = (p.tiles0 + p.tiles1) * p.ntiles;
    int splits = (sm_count + tiles - 1) / tiles;
    splits = max(1, min(splits, (ksteps + 3) / 4));
    const int per = (ksteps + splits - 1) / splits;
    p.kslice = per * kKStep;
    p.splits = (K + p.kslice - 1) / p.kslice;   // no empty split
    return p;
}

// GEMM C's plan: one split over K = rank.
Plan plan_gemm_c(const LayerParams& p, const LowRank& lr, int N, int sm_count) {
    Plan pc = plan_gemm(p.H * kHeadDim, 0, N, lr.rank, sm_count);
    pc.kslice = ((lr.rank + kKStep - 1) / kKStep) * kKStep;
    pc.splits = 1;
    return pc;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Scratch of one front-end call: GEMM A's partial sums, then u.
size_t scratch_bytes(const Plan& pa, int N, int rank) {
    return align256((size_t)pa.splits * N * pa.ldo * 4) + align256((size_t)N * rank * 4);
}

// Launch attributes for a kernel that may start before the one ahead of it
// in the stream has finished (programmatic dependent launch).
cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, cudaLaunchAttribute* attr,
                              bool pdl) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

cudaError_t run_gemm(const Plan& pl, const GemmMaps& maps, int N, int K, float* out, int* err_word,
                     cudaStream_t stream, bool pdl) {
    GemmArgs g{pl.tiles0, N, K, pl.Nt, pl.kslice, ring_stages(pl.Nt), pl.ldo, out};
    const dim3 grid((unsigned)(pl.tiles0 + pl.tiles1), (unsigned)pl.ntiles, (unsigned)pl.splits);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(grid, dim3(kThreads), gemm_smem_bytes(pl.Nt), stream, attr, pdl);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kda_lowrank_gemm_kernel, g, err_word, maps);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The three launches of one front-end call, with its scratch at `scratch`.
// GEMM A starts after everything before it in the stream; the reduction and
// GEMM C start early (programmatic dependent launch) and wait for their
// inputs inside, and so may a kernel launched that way after GEMM C.
cudaError_t run_frontend(const LayerParams& p, const LowRank& lr, const Plan& pa, int N, const float* x,
                         float* z, float* beta_logit, void* scratch, const DeviceInfo& dev, int* err_word,
                         cudaStream_t stream) {
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!g_attr_done[dev.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kda_lowrank_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)gemm_smem_bytes(256));
        if (e != cudaSuccess) return e;
        g_attr_done[dev.device].store(true, std::memory_order_release);
    }
    if (!lr.maps_ready) return cudaErrorInvalidValue;
    const int H = p.H;
    float* part = static_cast<float*>(scratch);
    float* u = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + align256((size_t)pa.splits * N * pa.ldo * 4));
    // GEMM A: [u | beta_logit] partial sums over the K splits.
    GemmMaps ma{};
    ma.a0 = lr.map_fa;
    ma.a1 = lr.map_bp;
    if (!make_map2d(&ma.b, x, lr.hidden, N, pa.Nt)) return cudaErrorInvalidValue;
    cudaError_t e = run_gemm(pa, ma, N, lr.hidden, part, err_word, stream, false);
    if (e != cudaSuccess) return e;
    // Reduce the splits.
    const size_t total = (size_t)N * (lr.rank + H);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg =
        pdl_config(dim3((unsigned)((total + 31) / 32)), dim3(32 * kReduceWarps), 0, stream, attr, true);
    e = cudaLaunchKernelEx(&cfg, kda_lowrank_reduce_kernel, (const float*)part, pa.splits, N, pa.ldo, lr.rank, H,
                           128 * pa.tiles0, u, beta_logit);
    count_launches(1);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
    // GEMM C: z = W_fb u, one split (K = rank).
    const Plan pc = plan_gemm_c(p, lr, N, dev.sm_count);
    GemmMaps mc{};
    mc.a0 = lr.map_fb;
    mc.a1 = lr.map_fb;
    if (!make_map2d(&mc.b, u, lr.rank, N, pc.Nt)) return cudaErrorInvalidValue;
    return run_gemm(pc, mc, N, lr.rank, z, err_word, stream, true);
}

}  // namespace

bool lowrank_prepare(const LayerParams& p, LowRank& lr) {
    lr.maps_ready = make_map2d(&lr.map_fa, lr.W_fa, lr.hidden, lr.rank, 128) &&
                    make_map2d(&lr.map_bp, lr.W_bp, lr.hidden, p.H, 128) &&
                    make_map2d(&lr.map_fb, lr.W_fb, lr.rank, p.H * kHeadDim, 128);
    return lr.maps_ready;
}

size_t lowrank_workspace_bytes(const LayerParams& p, const LowRank& lr, const DeviceInfo& dev, int N) {
    if (N <= 0) return 0;
    return scratch_bytes(plan_gemm(lr.rank, p.H, N, lr.hidden, dev.sm_count), N, lr.rank);
}

cudaError_t launch_lowrank(const LayerParams& p, const LowRank& lr, int N, const float* x, float* z,
                           float* beta_logit, void* workspace, const DeviceInfo& dev, int* err_word,
                           cudaStream_t stream) {
    if (N <= 0) return cudaSuccess;
    const Plan pa = plan_gemm(lr.rank, p.H, N, lr.hidden, dev.sm_count);
    return run_frontend(p, lr, pa, N, x, z, beta_logit, workspace, dev, err_word, stream);
}

// ---------------------------------------------------------------------------
// The front-end without a caller-supplied workspace (kda_lowrank_noalloc).
//
// Some callers cannot hand this library a workspace: a host runtime that
// passes a plugin only the tensors of the layer and owns every other byte of
// device memory, or a serving loop that must not allocate once it runs.  For
// them the front-end's scratch (the split-K partial sums and u) lives in one
// file-scope array of static device memory that comes with the library.
// Every GPU that loads the library holds the array until the process exits,
// so it is kept to KDA_LOWRANK_NOALLOC_SCRATCH_BYTES (4 MiB); a call whose
// scratch would not fit is rejected on the host.  All calls share the
// array: two calls that overlap on the GPU (different streams, or a second
// call before the first has finished on another stream) race on it.  It
// needs no clearing: every element a call reads was written earlier in the
// same call.
namespace {

static __device__ __align__(256) uint8_t g_lowrank_scratch[KDA_LOWRANK_NOALLOC_SCRATCH_BYTES];

// Host address of the array on each device, looked up once per device with
// that device current (the array's name in host code is only a stand-in).
struct ScratchAddr {
    std::once_flag once;
    void* ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
ScratchAddr g_scratch_addr[64];

// The plan of kda_lowrank, with the K split count lowered when the partial
// sums would not fit beside u in the static array.  Returns false when even
// one split does not fit.
bool plan_noalloc(const LayerParams& p, const LowRank& lr, const DeviceInfo& dev, int N, Plan* out,
                  size_t* need) {
    Plan pa = plan_gemm(lr.rank, p.H, N, lr.hidden, dev.sm_count);
    *need = scratch_bytes(pa, N, lr.rank);
    if (*need > (size_t)KDA_LOWRANK_NOALLOC_SCRATCH_BYTES) {
        const size_t ub = align256((size_t)N * lr.rank * 4);
        const size_t per_split = (size_t)N * pa.ldo * 4;
        const size_t room = (size_t)KDA_LOWRANK_NOALLOC_SCRATCH_BYTES > ub + 256
                                ? (size_t)KDA_LOWRANK_NOALLOC_SCRATCH_BYTES - ub - 256 : 0;
        const int cap = (int)(room / per_split);
        if (cap < 1) {
            pa.splits = 1;
            *need = scratch_bytes(pa, N, lr.rank);
            return false;
        }
        const int ksteps = (lr.hidden + kKStep - 1) / kKStep;
        const int per = (ksteps + cap - 1) / cap;
        pa.kslice = per * kKStep;
        pa.splits = (lr.hidden + pa.kslice - 1) / pa.kslice;
        *need = scratch_bytes(pa, N, lr.rank);
    }
    *out = pa;
    return true;
}

}  // namespace

size_t lowrank_noalloc_need(const LayerParams& p, const LowRank& lr, const DeviceInfo& dev, int N) {
    Plan pa;
    size_t need = 0;
    plan_noalloc(p, lr, dev, N, &pa, &need);
    return need;
}

cudaError_t launch_lowrank_noalloc(const LayerParams& p, const LowRank& lr, int N, const float* x, float* z,
                                   float* beta_logit, const DeviceInfo& dev, int* err_word, cudaStream_t stream) {
    if (N <= 0) return cudaSuccess;
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    ScratchAddr& sa = g_scratch_addr[dev.device];
    std::call_once(sa.once, [&] { sa.err = cudaGetSymbolAddress(&sa.ptr, g_lowrank_scratch); });
    if (sa.err != cudaSuccess) return sa.err;
    if (!sa.ptr) return cudaErrorInvalidSymbol;
    Plan pa;
    size_t need = 0;
    if (!plan_noalloc(p, lr, dev, N, &pa, &need)) return cudaErrorInvalidValue;   // the host checked the size
    return run_frontend(p, lr, pa, N, x, z, beta_logit, sa.ptr, dev, err_word, stream);
}

}  // namespace kda
