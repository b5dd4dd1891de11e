// Host side of the C ABI declared in include/kda.h: argument validation,
// device checks, launch and error reporting.  No allocation happens on the
// per-call path; kda_create allocates the 16-byte kernel error word.
//
// Fault injection for tests: KDA_FAULT_INJECT, read once by kda_create, is a
// comma-separated list of entry points ("decode", "prefill",
// "prefill_varlen", "lowrank", "project", or "all") whose launches that
// context replaces by the error cudaErrorLaunchFailure: nothing is launched,
// no buffer is touched and the call returns KDA_ERR_CUDA
// (kda_last_error_detail names the error and says it was injected).  The
// name "relay_drop" (not part of "all") instead makes kda_prefill's relay
// pairs skip their first state hand-over, and "split_drop" (not part of
// "all") makes the producers of its split schedule skip publishing their
// first chunk, so that a bounded wait inside the kernel runs out;
// "split_nofit" makes kda_prefill treat the split schedule's cooperative
// launch as not fitting on the device (it then runs the relay pairs).  Unset
// or empty: no injection.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "kda_internal.cuh"
#include "kda_testing.h"

struct kda_ctx {
    kda::LayerParams params;
    int chunk;
    kda::DeviceInfo dev;
    int* err_word;    // device int: nonzero after a kernel gave up on a bounded wait
    unsigned inject;  // launches replaced by an injected failure (KDA_FAULT_INJECT)
    bool has_lowrank;
    kda::LowRank lowrank;  // bound by kda_bind_lowrank
    bool has_proj;
    kda::Projections proj;  // bound by kda_bind_projections
};

namespace kda {
namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char g_detail[256] = "";

void set_detail(const char* what, cudaError_t e) {
    std::snprintf(g_detail, sizeof(g_detail), "%s: %s (%s)", what, cudaGetErrorName(e),
                  cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// A context is tied to the device current at kda_create: its kernels are
// launched on the current device, with the context's error word, so the two
// must agree.
kda_status check_device(const kda_ctx* ctx) {
    int cur = -1;
    const cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) { set_detail("cudaGetDevice", e); return KDA_ERR_CUDA; }
    if (cur != ctx->dev.device) {
        std::snprintf(g_detail, sizeof(g_detail), "current device %d is not the context's device %d",
                      cur, ctx->dev.device);
        return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

constexpr unsigned kInjectDecode = 1u, kInjectPrefill = 2u, kInjectVarlen = 4u, kInjectLowrank = 8u,
                   kInjectProject = 16u, kInjectRelayDrop = 32u,
                   kInjectSplitDrop = 64u, kInjectSplitNofit = 128u;

// Parse KDA_FAULT_INJECT (see the top of this file).
unsigned parse_inject(const char* v) {
    if (!v) return 0u;
    unsigned m = 0u;
    const char* p = v;
    while (*p) {
        const char* e = p;
        while (*e && *e != ',') ++e;
        const size_t n = (size_t)(e - p);
        auto is = [&](const char* w) { return std::strlen(w) == n && std::strncmp(p, w, n) == 0; };
        if (is("decode")) m |= kInjectDecode;
        else if (is("prefill")) m |= kInjectPrefill;
        else if (is("prefill_varlen")) m |= kInjectVarlen;
        else if (is("lowrank")) m |= kInjectLowrank;
        else if (is("project")) m |= kInjectProject;
        else if (is("relay_drop")) m |= kInjectRelayDrop;
        else if (is("split_drop")) m |= kInjectSplitDrop;
        else if (is("split_nofit")) m |= kInjectSplitNofit;
        else if (is("all")) m |= kInjectDecode | kInjectPrefill | kInjectVarlen | kInjectLowrank | kInjectProject;
        p = *e ? e + 1 : e;
    }
    return m;
}

// The launch itself, or the injected failure in its place.
template <typename F>
cudaError_t launch_or_inject(const kda_ctx* ctx, unsigned what, F&& launch) {
    if (ctx->inject & what) return cudaErrorLaunchFailure;
    return launch();
}

void set_launch_detail(const kda_ctx* ctx, unsigned what, const char* name, cudaError_t e) {
    if (ctx->inject & what) {
        std::snprintf(g_detail, sizeof(g_detail), "%s: %s (injected by KDA_FAULT_INJECT; nothing launched)",
                      name, cudaGetErrorName(e));
    } else {
        set_detail(name, e);
    }
}

}  // namespace

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace kda

using kda::aligned16;
using kda::aligned4;
using kda::check_device;

extern "C" {

const char* kda_strerror(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: null pointer, negative size or bad config";
        case KDA_ERR_ALIGNMENT: return "KDA_ERR_ALIGNMENT: a pointer is not 16-byte (beta_logit: 4-byte) aligned";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: head_dim must be 128, chunk_size 64, device sm_103";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call failed (see kda_last_error_detail)";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
    }
    return "unknown kda_status";
}

const char* kda_last_error_detail(void) { return kda::g_detail; }

uint64_t kda_launch_count(void) { return kda::g_launches.load(std::memory_order_relaxed); }

kda_status kda_create(const kda_config* cfg, const float* conv_w, const float* dt_bias,
                      const float* A_log, const float* rms_gamma, kda_ctx** out) {
    if (!out) return KDA_ERR_INVALID_ARG;
    *out = nullptr;
    if (!cfg || !conv_w || !dt_bias || !A_log || !rms_gamma) return KDA_ERR_INVALID_ARG;
    if (cfg->num_heads < 1 || !(cfg->l2_eps >= 0.0f) || !(cfg->rms_eps >= 0.0f) ||
        !std::isfinite(cfg->l2_eps) || !std::isfinite(cfg->rms_eps))
        return KDA_ERR_INVALID_ARG;
    if (cfg->head_dim != kda::kHeadDim || cfg->chunk_size != kda::kChunk) return KDA_ERR_UNSUPPORTED;
    if (!aligned16(conv_w) || !aligned16(dt_bias) || !aligned16(A_log) || !aligned16(rms_gamma))
        return KDA_ERR_ALIGNMENT;

    kda::DeviceInfo dev{};
    cudaError_t e = cudaGetDevice(&dev.device);
    if (e != cudaSuccess) { kda::set_detail("cudaGetDevice", e); return KDA_ERR_CUDA; }
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev.device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev.device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&dev.sm_count, cudaDevAttrMultiProcessorCount, dev.device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&dev.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    dev.device)) != cudaSuccess) {
        kda::set_detail("cudaDeviceGetAttribute", e);
        return KDA_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail),
                      "device %d is sm_%d%d; this library is built for sm_103a only", dev.device,
                      major, minor);
        return KDA_ERR_UNSUPPORTED;
    }
    kda_ctx* c = new (std::nothrow) kda_ctx{};
    if (!c) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail), "host allocation of the context failed");
        return KDA_ERR_INVALID_ARG;
    }
    c->params = kda::LayerParams{cfg->num_heads, cfg->l2_eps, cfg->rms_eps,
                                 conv_w, dt_bias, A_log, rms_gamma};
    c->chunk = cfg->chunk_size;
    c->dev = dev;
    c->inject = kda::parse_inject(std::getenv("KDA_FAULT_INJECT"));
    if ((e = cudaMalloc(&c->err_word, 16)) != cudaSuccess) {
        kda::set_detail("cudaMalloc(error word)", e);
        delete c;
        return KDA_ERR_CUDA;
    }
    if ((e = cudaMemset(c->err_word, 0, 16)) != cudaSuccess) {
        kda::set_detail("cudaMemset(error word)", e);
        cudaFree(c->err_word);
        delete c;
        return KDA_ERR_CUDA;
    }
    *out = c;
    return KDA_OK;
}

void kda_destroy(kda_ctx* ctx) {
    if (!ctx) return;
    if (ctx->err_word) cudaFree(ctx->err_word);
    delete ctx;
}

kda_status kda_decode_step(kda_ctx* ctx, int B, const float* q, const float* k, const float* v,
                           const float* z, const float* beta_logit, const float* gate_logit,
                           float* conv_state, float* S, float* o, float* o_pre, void* stream) {
    if (!ctx || B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !z || !beta_logit || !gate_logit || !conv_state || !S || !o)
        return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, z, gate_logit, conv_state, S, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (!aligned4(beta_logit)) return KDA_ERR_ALIGNMENT;
    if (o_pre && !aligned16(o_pre)) return KDA_ERR_ALIGNMENT;
    if ((long long)B * ctx->params.H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    kda::DecodeIO io{B, q, k, v, z, beta_logit, gate_logit, conv_state, S, o, o_pre};
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectDecode, [&] {
        return kda::launch_decode(ctx->params, io, ctx->dev, ctx->err_word, static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) { kda::set_launch_detail(ctx, kda::kInjectDecode, "decode launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

kda_status kda_decode_step_bf16state(kda_ctx* ctx, int B, const float* q, const float* k, const float* v,
                                     const float* z, const float* beta_logit, const float* gate_logit,
                                     float* conv_state, uint16_t* S, float* o, float* o_pre, void* stream) {
    if (!ctx || B < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !z || !beta_logit || !gate_logit || !conv_state || !S || !o)
        return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, z, gate_logit, conv_state, S, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (!aligned4(beta_logit)) return KDA_ERR_ALIGNMENT;
    if (o_pre && !aligned16(o_pre)) return KDA_ERR_ALIGNMENT;
    if ((long long)B * ctx->params.H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    kda::DecodeIO io{B, q, k, v, z, beta_logit, gate_logit, conv_state, nullptr, o, o_pre, S};
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectDecode, [&] {
        return kda::launch_decode(ctx->params, io, ctx->dev, ctx->err_word, static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) { kda::set_launch_detail(ctx, kda::kInjectDecode, "decode launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

size_t kda_prefill_workspace_bytes(const kda_ctx* ctx, int B, int T) {
    if (!ctx || B <= 0 || T <= 0) return 0;
    return kda::prefill_workspace_bytes(ctx->params.H, B, T, ctx->dev);
}

kda_status kda_prefill(kda_ctx* ctx, int B, int T, const uint16_t* q, const uint16_t* k,
                       const uint16_t* v, const float* z, const float* beta_logit,
                       const float* gate_logit, float* conv_state, float* S, float* o,
                       void* workspace, size_t workspace_bytes, void* stream) {
    if (!ctx || B < 0 || T < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0 || T == 0) return KDA_OK;
    if (!q || !k || !v || !z || !beta_logit || !gate_logit || !conv_state || !S || !o)
        return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, z, gate_logit, conv_state, S, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (!aligned4(beta_logit)) return KDA_ERR_ALIGNMENT;
    if ((long long)B * ctx->params.H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    // The workspace is optional: with kda_prefill_workspace_bytes of it the
    // few-head schedule splits producers from consumers, else it runs relay pairs.
    if (workspace && !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
    if (!workspace) workspace_bytes = 0;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    kda::PrefillIO io{B, T, nullptr, q, k, v, z, beta_logit, gate_logit, conv_state, S, o,
                      workspace, workspace_bytes, 0, (ctx->inject & kda::kInjectRelayDrop) ? 1 : 0,
                      (ctx->inject & kda::kInjectSplitDrop) ? 1 : 0, (ctx->inject & kda::kInjectSplitNofit) ? 1 : 0};
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectPrefill, [&] {
        return kda::launch_prefill(ctx->params, io, ctx->dev, ctx->err_word, static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) { kda::set_launch_detail(ctx, kda::kInjectPrefill, "prefill launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

kda_status kda_prefill_varlen(kda_ctx* ctx, int B, const int32_t* cu_seqlens, int total_T,
                              const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* z,
                              const float* beta_logit, const float* gate_logit, float* conv_state,
                              float* S, float* o, void* stream) {
    if (!ctx || B < 0 || total_T < 0) return KDA_ERR_INVALID_ARG;
    if (B == 0 || total_T == 0) return KDA_OK;   // every sequence empty: state and window unchanged
    if (!cu_seqlens || !q || !k || !v || !z || !beta_logit || !gate_logit || !conv_state || !S || !o)
        return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, z, gate_logit, conv_state, S, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (!aligned4(beta_logit) || !aligned4(cu_seqlens)) return KDA_ERR_ALIGNMENT;
    if ((long long)B * ctx->params.H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    kda::PrefillIO io{B, total_T, cu_seqlens, q, k, v, z, beta_logit, gate_logit, conv_state, S, o,
                      nullptr, 0, 0};
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectVarlen, [&] {
        return kda::launch_prefill(ctx->params, io, ctx->dev, ctx->err_word, static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) { kda::set_launch_detail(ctx, kda::kInjectVarlen, "prefill_varlen launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

kda_status kda_sync_status(kda_ctx* ctx, void* stream) {
    if (!ctx) return KDA_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { kda::set_detail("cudaStreamSynchronize", e); return KDA_ERR_CUDA; }
    int word = 0;
    if ((e = cudaMemcpy(&word, ctx->err_word, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) {
        kda::set_detail("cudaMemcpy(error word)", e);
        return KDA_ERR_CUDA;
    }
    if (word != 0) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail),
                      "kernel error word 0x%x (bounded wait gave up)", word);
        if ((e = cudaMemset(ctx->err_word, 0, sizeof(int))) != cudaSuccess) {
            kda::set_detail("cudaMemset(error word)", e);
            return KDA_ERR_CUDA;
        }
        return KDA_ERR_TIMEOUT;
    }
    return KDA_OK;
}

kda_status kda_bind_lowrank(kda_ctx* ctx, int hidden, int rank, const float* W_fa, const float* W_fb,
                            const float* W_bp) {
    if (!ctx || !W_fa || !W_fb || !W_bp) return KDA_ERR_INVALID_ARG;
    if (hidden < 4 || rank < 4 || rank > 512 || (hidden & 3) || (rank & 3)) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail),
                      "hidden (%d) and rank (%d) must be multiples of 4, rank at most 512", hidden, rank);
        return KDA_ERR_INVALID_ARG;
    }
    if (!aligned16(W_fa) || !aligned16(W_fb) || !aligned16(W_bp)) return KDA_ERR_ALIGNMENT;
    kda::LowRank lr{};
    lr.hidden = hidden;
    lr.rank = rank;
    lr.W_fa = W_fa;
    lr.W_fb = W_fb;
    lr.W_bp = W_bp;
    if (!kda::lowrank_prepare(ctx->params, lr)) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail), "cuTensorMapEncodeTiled failed for the low-rank weights");
        return KDA_ERR_CUDA;
    }
    ctx->lowrank = lr;
    ctx->has_lowrank = true;
    return KDA_OK;
}

size_t kda_lowrank_workspace_bytes(const kda_ctx* ctx, int N) {
    if (!ctx || !ctx->has_lowrank || N <= 0) return 0;
    return kda::lowrank_workspace_bytes(ctx->params, ctx->lowrank, ctx->dev, N);
}

kda_status kda_lowrank(kda_ctx* ctx, int N, const float* x, float* z, float* beta_logit, void* workspace,
                       size_t workspace_bytes, void* stream) {
    if (!ctx || N < 0) return KDA_ERR_INVALID_ARG;
    if (!ctx->has_lowrank) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail), "no low-rank weights bound (kda_bind_lowrank)");
        return KDA_ERR_INVALID_ARG;
    }
    if (N == 0) return KDA_OK;
    if (!x || !z || !beta_logit || !workspace) return KDA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(z) || !aligned4(beta_logit) || !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
    if (workspace_bytes < kda::lowrank_workspace_bytes(ctx->params, ctx->lowrank, ctx->dev, N))
        return KDA_ERR_INVALID_ARG;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectLowrank, [&] {
        return kda::launch_lowrank(ctx->params, ctx->lowrank, N, x, z, beta_logit, workspace, ctx->dev,
                                   ctx->err_word, static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) { kda::set_launch_detail(ctx, kda::kInjectLowrank, "lowrank launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

kda_status kda_lowrank_noalloc(kda_ctx* ctx, int N, const float* x, float* z, float* beta_logit, void* stream) {
    if (!ctx || N < 0) return KDA_ERR_INVALID_ARG;
    if (!ctx->has_lowrank) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail), "no low-rank weights bound (kda_bind_lowrank)");
        return KDA_ERR_INVALID_ARG;
    }
    if (N == 0) return KDA_OK;
    if (!x || !z || !beta_logit) return KDA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(z) || !aligned4(beta_logit)) return KDA_ERR_ALIGNMENT;
    const size_t need = kda::lowrank_noalloc_need(ctx->params, ctx->lowrank, ctx->dev, N);
    if (need > (size_t)KDA_LOWRANK_NOALLOC_SCRATCH_BYTES) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail),
                      "kda_lowrank_noalloc: %d tokens need %zu bytes of scratch, more than its static %u-byte array",
                      N, need, (unsigned)KDA_LOWRANK_NOALLOC_SCRATCH_BYTES);
        return KDA_ERR_INVALID_ARG;
    }
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectLowrank, [&] {
        return kda::launch_lowrank_noalloc(ctx->params, ctx->lowrank, N, x, z, beta_logit, ctx->dev, ctx->err_word,
                                           static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) {
        kda::set_launch_detail(ctx, kda::kInjectLowrank, "lowrank_noalloc launch", e);
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

// Workspace of kda_decode_step_lowrank: the front-end's own, then z [B][H][d]
// and beta_logit [B][H].
static size_t decode_lowrank_parts(const kda_ctx* ctx, int B, size_t* off_z, size_t* off_b) {
    const size_t a = (kda::lowrank_workspace_bytes(ctx->params, ctx->lowrank, ctx->dev, B) + 255) & ~size_t(255);
    const size_t zb = (size_t)B * ctx->params.H * kda::kHeadDim * 4;
    *off_z = a;
    *off_b = (a + zb + 255) & ~size_t(255);
    return *off_b + (size_t)B * ctx->params.H * 4;
}

size_t kda_decode_lowrank_workspace_bytes(const kda_ctx* ctx, int B) {
    if (!ctx || !ctx->has_lowrank || B <= 0) return 0;
    size_t oz, ob;
    return decode_lowrank_parts(ctx, B, &oz, &ob);
}

kda_status kda_decode_step_lowrank(kda_ctx* ctx, int B, const float* x, const float* q, const float* k,
                                   const float* v, const float* gate_logit, float* conv_state, float* S,
                                   float* o, float* o_pre, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    if (!ctx || B < 0) return KDA_ERR_INVALID_ARG;
    if (!ctx->has_lowrank) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail), "no low-rank weights bound (kda_bind_lowrank)");
        return KDA_ERR_INVALID_ARG;
    }
    if (B == 0) return KDA_OK;
    if (!x || !q || !k || !v || !gate_logit || !conv_state || !S || !o || !workspace) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {x, q, k, v, gate_logit, conv_state, S, o, workspace};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (o_pre && !aligned16(o_pre)) return KDA_ERR_ALIGNMENT;
    if ((long long)B * ctx->params.H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    size_t oz, ob;
    if (workspace_bytes < decode_lowrank_parts(ctx, B, &oz, &ob)) return KDA_ERR_INVALID_ARG;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    float* z = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + oz);
    float* bl = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ob);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectLowrank | kda::kInjectDecode, [&] {
        cudaError_t r = kda::launch_lowrank(ctx->params, ctx->lowrank, B, x, z, bl, workspace, ctx->dev,
                                            ctx->err_word, st);
        if (r != cudaSuccess) return r;
        kda::DecodeIO io{B, q, k, v, z, bl, gate_logit, conv_state, S, o, o_pre};
        return kda::launch_decode(ctx->params, io, ctx->dev, ctx->err_word, st, true);
    });
    if (e != cudaSuccess) {
        kda::set_launch_detail(ctx, kda::kInjectLowrank | kda::kInjectDecode, "decode_lowrank launch", e);
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

kda_status kda_bind_projections(kda_ctx* ctx, int hidden, const uint16_t* W_qkvg, const uint16_t* W_o) {
    if (!ctx || !W_qkvg || !W_o) return KDA_ERR_INVALID_ARG;
    if (hidden < 128 || hidden % 128) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail), "hidden (%d) must be a positive multiple of 128", hidden);
        return KDA_ERR_INVALID_ARG;
    }
    if (!aligned16(W_qkvg) || !aligned16(W_o)) return KDA_ERR_ALIGNMENT;
    kda::Projections pr{};
    pr.hidden = hidden;
    pr.W_qkvg = W_qkvg;
    pr.W_o = W_o;
    if (!kda::proj_prepare(ctx->params, pr)) {
        std::snprintf(kda::g_detail, sizeof(kda::g_detail), "cuTensorMapEncodeTiled failed for the projection weights");
        return KDA_ERR_CUDA;
    }
    ctx->proj = pr;
    ctx->has_proj = true;
    return KDA_OK;
}

static kda_status need_proj(const kda_ctx* ctx) {
    if (ctx->has_proj) return KDA_OK;
    std::snprintf(kda::g_detail, sizeof(kda::g_detail), "no projection weights bound (kda_bind_projections)");
    return KDA_ERR_INVALID_ARG;
}

kda_status kda_project_qkvg(kda_ctx* ctx, int N, const uint16_t* x, void* q, void* k, void* v, float* gate_logit,
                            int qkv_f32, void* stream) {
    if (!ctx || N < 0) return KDA_ERR_INVALID_ARG;
    if (const kda_status r = need_proj(ctx); r != KDA_OK) return r;
    if (N == 0) return KDA_OK;
    if (!x || !q || !k || !v || !gate_logit) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {x, q, k, v, gate_logit};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectProject, [&] {
        return kda::launch_project_qkvg(ctx->params, ctx->proj, N, x, q, k, v, gate_logit, qkv_f32 != 0, ctx->dev,
                                        ctx->err_word, static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) { kda::set_launch_detail(ctx, kda::kInjectProject, "project_qkvg launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

size_t kda_project_o_workspace_bytes(const kda_ctx* ctx, int N) {
    if (!ctx || N <= 0) return 0;
    return kda::project_o_workspace_bytes(ctx->params, N);
}

kda_status kda_project_o(kda_ctx* ctx, int N, const float* o, float* y, void* workspace, size_t workspace_bytes,
                         void* stream) {
    if (!ctx || N < 0) return KDA_ERR_INVALID_ARG;
    if (const kda_status r = need_proj(ctx); r != KDA_OK) return r;
    if (N == 0) return KDA_OK;
    if (!o || !y || !workspace) return KDA_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(y) || !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
    if (workspace_bytes < kda::project_o_workspace_bytes(ctx->params, N)) return KDA_ERR_INVALID_ARG;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    cudaError_t e = kda::launch_or_inject(ctx, kda::kInjectProject, [&] {
        return kda::launch_project_o(ctx->params, ctx->proj, N, o, y, workspace, ctx->dev, ctx->err_word,
                                     static_cast<cudaStream_t>(stream));
    });
    if (e != cudaSuccess) { kda::set_launch_detail(ctx, kda::kInjectProject, "project_o launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

kda_status kda_testing_bounded_wait(kda_ctx* ctx, unsigned limit_us, void* stream) {
    if (!ctx || limit_us < 1 || limit_us > 1000000) return KDA_ERR_INVALID_ARG;
    if (const kda_status d = check_device(ctx); d != KDA_OK) return d;
    cudaError_t e = kda::launch_testing_wait(ctx->err_word, 1000ull * limit_us, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { kda::set_detail("testing wait launch", e); return KDA_ERR_CUDA; }
    return KDA_OK;
}

long long kda_testing_prefill_relay_heads(long long heads, int T, int sm_count) {
    if (heads < 0 || T < 0 || sm_count < 0) return -1;
    return kda::prefill_relay_heads(heads, T, sm_count);
}

int kda_testing_project_o_ksplit(int hidden, int N, int HD, int sm_count) {
    if (hidden < 0 || N <= 0 || HD < 0 || sm_count < 0) return -1;
    return kda::project_o_ksplit(hidden, N, HD, sm_count);
}

}  // extern "C"
