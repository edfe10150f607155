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

// (cos, sin) of the angle of pair index d at position pos: a kernel may compute them
// once per pair index and reuse them for every head.
__device__ __forceinline__ float2 rope_cos_sin(int pos, float inv_freq) {
    float s, c;
    sincosf(rope_theta(pos, inv_freq), &s, &c);
    return make_float2(c, s);
}

// Neox rotation of the pair (x0, x1) = (element d, element d + hd/2) by the angle with
// cos cs.x and sin cs.y: (x0 cos - x1 sin, x0 sin + x1 cos).
__device__ __forceinline__ void rope_rotate_cs(float x0, float x1, float2 cs, float& r0, float& r1) {
    r0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
    r1 = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
}

__device__ __forceinline__ void rope_rotate(float x0, float x1, float theta, float& r0, float& r1) {
    float s, c;
    sincosf(theta, &s, &c);
    rope_rotate_cs(x0, x1, make_float2(c, s), r0, r1);
}

// Cache element store at flat index pos * nkt + j (f32, or f16 round-to-nearest-even).
__device__ __forceinline__ void kv_put(void* kv, int f16, size_t idx, float v) {
    if (f16) reinterpret_cast<__half*>(kv)[idx] = __float2half_rn(v);
    else reinterpret_cast<float*>(kv)[idx] = v;
}

__device__ __forceinline__ bool pos_ok(int pos, int n_ctx) { return pos >= 0 && pos < n_ctx; }

}  // namespace qkv_epi
