// Internal declarations shared by the host API and the kernels of the CUDA
// library.  Nothing here is part of the public C ABI (include/kda.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kHeadDim = 128;   // d_k = d_v
constexpr int kChunk = 64;      // prefill chunk length

// Everything a kernel needs about one layer: borrowed parameter pointers and
// the normalisation epsilons.  Passed by value as a kernel argument.
struct LayerParams {
    int H;
    float l2_eps;
    float rms_eps;
    const float* conv_w;   // [3][H*d][4]
    const float* dt_bias;  // [H][d]
    const float* A_log;    // [H][d]
    const float* gamma;    // [H][d]
};

struct DecodeIO {
    int B;
    const float* q;
    const float* k;
    const float* v;
    const float* z;
    const float* beta_logit;
    const float* gate_logit;
    float* conv_state;
    float* S;
    float* o;
    float* o_pre;  // may be null
    uint16_t* S16; // bf16 state instead of S (then S is null), or null
};

struct PrefillIO {
    int B;
    int T;              // tokens per sequence, or the total of packed sequences
    const int* cu_seqlens;   // null, or [B + 1] device offsets of packed sequences
    const uint16_t* q;  // bf16 bits
    const uint16_t* k;
    const uint16_t* v;
    const float* z;
    const float* beta_logit;
    const float* gate_logit;
    float* conv_state;
    float* S;
    float* o;
    void* workspace;
    size_t workspace_bytes;
    // Relay launches (set by launch_prefill): heads [head0, head0 + grid/2)
    // run as clusters of two CTAs that take alternate chunks and hand the
    // state over through distributed shared memory.
    int head0;
    // Test injection (KDA_FAULT_INJECT "relay_drop"): the first CTA of every
    // relay pair does not hand its first state over, so the second one's
    // bounded wait runs out.
    int drop_relay;
    // Test injection (KDA_FAULT_INJECT "split_drop"): the producers of the
    // split schedule do not publish their first chunk, so its consumer's
    // bounded wait runs out.
    int drop_split;
    // Test injection (KDA_FAULT_INJECT "split_nofit"): the split schedule's
    // cooperative launch is treated as not fitting on the device, so the
    // relay pairs run instead.
    int nofit_split;
};

// Low-rank front-end weights bound to a context (borrowed, fp32), with
// their TMA tensor maps (encoded once, at binding, by lowrank_prepare).
struct LowRank {
    int hidden;           // width of the hidden input x
    int rank;             // inner width of W_fb W_fa
    const float* W_fa;    // [rank][hidden]
    const float* W_fb;    // [H*d][rank]
    const float* W_bp;    // [H][hidden]
    bool maps_ready;
    CUtensorMap map_fa, map_bp, map_fb;
};

// Projection weights bound to a context (borrowed, bf16), with their TMA
// tensor maps (encoded once, at binding, by proj_prepare).
struct Projections {
    int hidden;             // width of the hidden input x and of y
    const void* W_qkvg;     // [4*H*d][hidden] bf16: W_q, W_k, W_v, W_g stacked by rows
    const void* W_o;        // [hidden][H*d] bf16
    bool maps_ready;
    CUtensorMap map_qkvg, map_o;
};

// Device facts the launchers need, queried once per context.
struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
};

// Launchers (kernels live in decode.cu / prefill.cu).  They return the
// cudaError_t of the launch.
// pdl: the kernel may start while the kernel before it in the stream (the
// low-rank front-end) finishes; it waits for that kernel before reading z and
// beta_logit.
cudaError_t launch_decode(const LayerParams& p, const DecodeIO& io, const DeviceInfo& dev,
                          int* err_word, cudaStream_t stream, bool pdl = false);
size_t prefill_workspace_bytes(int H, int B, int T, const DeviceInfo& dev);
cudaError_t launch_prefill(const LayerParams& p, const PrefillIO& io, const DeviceInfo& dev,
                           int* err_word, cudaStream_t stream);

// Low-rank front-end (csrc/lowrank.cu): z [N][H*d] and beta_logit [N][H] of
// N tokens of hidden input x [N][hidden]; workspace of lowrank_workspace_bytes.
// lowrank_prepare encodes the weights' tensor maps (false if it cannot).
bool lowrank_prepare(const LayerParams& p, LowRank& lr);
size_t lowrank_workspace_bytes(const LayerParams& p, const LowRank& lr, const DeviceInfo& dev, int N);
cudaError_t launch_lowrank(const LayerParams& p, const LowRank& lr, int N, const float* x, float* z,
                           float* beta_logit, void* workspace, const DeviceInfo& dev, int* err_word,
                           cudaStream_t stream);

// The front-end with its scratch in a static device array (csrc/lowrank.cu):
// bytes of that array a call for N tokens needs (more than
// KDA_LOWRANK_NOALLOC_SCRATCH_BYTES: the call cannot run), and the launch.
size_t lowrank_noalloc_need(const LayerParams& p, const LowRank& lr, const DeviceInfo& dev, int N);
cudaError_t launch_lowrank_noalloc(const LayerParams& p, const LowRank& lr, int N, const float* x, float* z,
                                   float* beta_logit, const DeviceInfo& dev, int* err_word, cudaStream_t stream);

// Projections (csrc/proj.cu): input projections of N tokens of bf16 x into
// q, k, v (bf16, or fp32 when qkv_f32) and fp32 gate logits; output
// projection of fp32 o into fp32 y through a bf16 copy of o in `workspace`
// (project_o_workspace_bytes).
bool proj_prepare(const LayerParams& p, Projections& pr);
cudaError_t launch_project_qkvg(const LayerParams& p, const Projections& pr, int N, const void* x, void* q,
                                void* k, void* v, float* gate_logit, bool qkv_f32, const DeviceInfo& dev,
                                int* err_word, cudaStream_t stream);
size_t project_o_workspace_bytes(const LayerParams& p, int N);
cudaError_t launch_project_o(const LayerParams& p, const Projections& pr, int N, const float* o, float* y,
                             void* workspace, const DeviceInfo& dev, int* err_word, cudaStream_t stream);

// Test hook (csrc/testing.cu): a kernel whose bounded wait runs out.
cudaError_t launch_testing_wait(int* err_word, unsigned long long limit_ns, cudaStream_t stream);

// Launch policies (exported through the test hooks): how many of `heads`
// (sequence, head) pairs of a T-token prefill run as relay pairs on a
// device of sm_count SMs, and into how many K ranges the output projection
// of N tokens (hidden outputs, HD inputs) is split.
long long prefill_relay_heads(long long heads, int T, int sm_count);
int project_o_ksplit(int hidden, int N, int HD, int sm_count);

// Counts kernel launches made by the library (for benchmark accounting).
void count_launches(uint64_t n);

}  // namespace kda
