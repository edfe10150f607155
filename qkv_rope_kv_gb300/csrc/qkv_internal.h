// Internal declarations shared by the C-ABI layer and the kernel files of
// libqkv.so.  Not part of the public interface (include/qkv.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "qkv.h"

struct qkv_plan {
    qkv_plan_desc d;
    int64_t nqt, nkt, rows, half;
    int vec;  // rows can be streamed as aligned 16-byte vectors (H * elem % 16 == 0)
    float inv_freq[QKV_MAX_HEAD_DIM / 2];
};

// Everything one decode-layer launch needs, passed by value (__grid_constant__),
// so a captured graph node carries its own copy.
struct DecodeParams {
    const float* x;         // [H] hidden vector
    const void* w[3];       // q / k / v weight sections, row-major [rows x H]
    const float* bias[3];   // q / k / v bias sections (fused and epilogue modes)
    float* out[3];          // q / k / v outputs (in-place epilogue operands)
    void* kv_k;             // K region [n_ctx x nkt]
    void* kv_v;             // V region [n_ctx x nkt]
    const int32_t* pos;     // device position
    int32_t H, nqt, nkt, hd, n_ctx, kv_f16;
    int32_t nf;             // FusedFFN: rows per half of the gate|up weight (0 for the QKV stage)
    const float* norm_w;    // RMSNorm weight [H]: x is then the hidden state h, normalised in-kernel
    float norm_eps;         // RMSNorm epsilon
    const float* qk_norm_w[2];  // FusedQkvNorm: per-head norm weights of q and k [hd] each
    float qk_eps;               // FusedQkvNorm epsilon
    unsigned int* head_cnt;     // FusedQkvNorm: per-head completion counters [nh + nkv], zero between launches
    // Weight sections of the next layer of a model graph when it has this layer's shape, else
    // null: a read-only L2 prefetch hint (the pair ring brings its first items into L2 while
    // this layer finishes); no result depends on it.
    const void* next_w[3];
    // Test hook of the bounded waits (zero in every product call): a non-zero wait limit
    // replaces the default, and withhold_last_copy makes the ring producers skip each
    // CTA's last weight copy, so the wait for it runs out.
    unsigned long long wait_limit_ns;
    int32_t withhold_last_copy;
    float inv_freq[QKV_MAX_HEAD_DIM / 2];
};

enum DecodeMode { kProjectOnly = 0, kFused = 1 };

// decode_kernels.cu
cudaError_t launch_decode(const DecodeParams& p, int w_dtype, int vec, DecodeMode mode, bool pdl,
                          cudaStream_t stream);
cudaError_t launch_epilogue(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_chain_add_bias(float* y, const float* b, int64_t n, cudaStream_t stream);
cudaError_t launch_chain_rope(const DecodeParams& p, float* y, int n_heads, cudaStream_t stream);
cudaError_t launch_chain_store(const DecodeParams& p, const float* src, void* cache,
                               cudaStream_t stream);
cudaError_t device_status_read(cudaStream_t stream, uint32_t* flags, int32_t* bad_pos);
// FusedFFN decode: out[i] = silu((W x)[i]) * (W x)[nf + i] over the concat gate|up
// weight p.w[0] [2 nf x H] into p.out[0] [nf]; rows must be 16-byte aligned.
// Returns cudaErrorNotSupported when no ring shape fits the hidden size.
cudaError_t launch_ffn(const DecodeParams& p, int w_dtype, bool pdl, cudaStream_t stream);
// FusedQkvNorm decode: the fused stage with each q and k head RMS-normalised (weights
// p.qk_norm_w, epsilon p.qk_eps) after its bias and before its rotation; p.head_cnt is a
// zeroed workspace of nh + nkv counters, left zeroed.  Rows must be 16-byte aligned.
// Returns cudaErrorNotSupported when no ring shape fits the hidden size.
cudaError_t launch_qknorm(const DecodeParams& p, int w_dtype, bool pdl, cudaStream_t stream);
// The library's own FusedQkvNorm counters (a fixed device array of kQknormStaticHeads
// entries): their device address on the current device, looked up on first use there.
constexpr int kQknormStaticHeads = 1024;
constexpr int kQknormMaxDevices = 64;
cudaError_t qknorm_static_workspace(unsigned int** out);

// prefill_tcgen05.cu
struct PrefillParams {
    const uint16_t* X;      // [nt x H] bf16
    const uint16_t* W;      // [R x H] bf16
    const float* bias;      // [R]
    const int32_t* positions;
    float* Y;               // [nt x R]
    void* kv_k;
    void* kv_v;
    int32_t nt, H, nqt, nkt, hd, n_ctx, kv_f16;
    // Test hook of the bounded waits (zero in every product call): a non-zero wait limit
    // replaces the default, and withhold_xchg makes each CTA of a cluster of 2 skip sending its
    // partial sums to the peer, so the peer's wait for them runs out.
    unsigned long long wait_limit_ns;
    int32_t withhold_xchg;
    float inv_freq[QKV_MAX_HEAD_DIM / 2];
};
qkv_status launch_prefill(const PrefillParams& p, bool pdl, cudaStream_t stream, const char** why);
cudaError_t prefill_status_read(cudaStream_t stream, uint32_t* flags, int32_t* bad_pos);
