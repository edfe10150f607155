// Per-element epilogue math of the attention-input stage, shared by every
// kernel that finishes a projection (decode fused tail, one-launch epilogue,
// seven-launch chain, prefill GEMM epilogue), so that all of them produce the
// same bits for the same f32 inputs ("73 · D3-8 — G4 FusedQKV ported to CUDA",
// §2, "The fusion's bitwise legitimacy").  Explicit _rn intrinsics: no FMA
// contraction can differ between call sites.
#pragma once

#include <cuda_fp16.h>
#include <stddef.h>

namespace qkv_epi {

// Angle of pair index d at position pos: the f32 product pos * inv_freq[d]
// (§3.2 Excerpt A: theta = pos * freq).
__device__ __forceinline__ float rope_theta(int pos, float inv_freq) {
    return __fmul_rn(__int2float_rn(pos), inv_freq);
}

// Neox rotation of the pair (x0, x1) = (element d, element d + hd/2):
// (x0 cos - x1 sin, x0 sin + x1 cos).
__device__ __forceinline__ void rope_rotate(float x0, float x1, float theta, float& r0, float& r1) {
    float s, c;
    sincosf(theta, &s, &c);
    r0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    r1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
}

// Cache element store at flat index pos * nkt + j (f32, or f16 round-to-nearest-even).
__device__ __forceinline__ void kv_put(void* kv, int f16, size_t idx, float v) {
    if (f16) reinterpret_cast<__half*>(kv)[idx] = __float2half_rn(v);
    else reinterpret_cast<float*>(kv)[idx] = v;
}

__device__ __forceinline__ bool pos_ok(int pos, int n_ctx) { return pos >= 0 && pos < n_ctx; }

}  // namespace qkv_epi
