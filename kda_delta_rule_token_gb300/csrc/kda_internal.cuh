// Internal declarations shared by the host API and the kernels of the CUDA
// library.  Nothing here is part of the public C ABI (include/kda.h).
#pragma once

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
};

// Device facts the launchers need, queried once per context.
struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
};

// Launchers (kernels live in decode.cu / prefill.cu).  They return the
// cudaError_t of the launch.
cudaError_t launch_decode(const LayerParams& p, const DecodeIO& io, const DeviceInfo& dev,
                          int* err_word, cudaStream_t stream);
size_t prefill_workspace_bytes(int H, int B, int T);
cudaError_t launch_prefill(const LayerParams& p, const PrefillIO& io, const DeviceInfo& dev,
                           int* err_word, cudaStream_t stream);

// Test hook (csrc/testing.cu): a kernel whose bounded wait runs out.
cudaError_t launch_testing_wait(int* err_word, unsigned long long limit_ns, cudaStream_t stream);

// Counts kernel launches made by the library (for benchmark accounting).
void count_launches(uint64_t n);

}  // namespace kda
