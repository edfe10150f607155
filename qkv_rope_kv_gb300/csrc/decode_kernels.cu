// Decode (nt == 1) kernels of the attention-input stage on sm_103a.
//
//   qkv_decode_blk_kernel  block ring, rows of >= 8 KB (the 14B shape): persistent
//                          CTAs, one per SM; a producer lane streams blocks of
//                          two adjacent rows into a shared-memory ring with
//                          cp.async.bulk, five one-warp consumer groups reduce
//                          them and finish each unit's neox pairs (bias, RoPE,
//                          KV-cache store).  The same ring runs the FusedFFN
//                          (silu(gate) * up) and the FusedQkvNorm stage.
//   qkv_decode_tma_kernel  pair ring, shorter 16-byte aligned rows (7B, 0.5B):
//                          one neox pair (two copies) per stage; two CTAs per
//                          SM with three consumer groups (rows of 4-8 KB), or
//                          three with two groups (rows under 4 KB).
//   qkv_decode_kernel      register streaming, one row pair per warp with
//                          16-byte non-allocating loads: rows that are not
//                          16-byte aligned or too long to stage.
//   qkv_epilogue_kernel    the epilogue alone over the flat index
//                          nqt/2 + nkt/2 + nkt ("73 · D3-8 — G4 FusedQKV ported
//                          to CUDA", §3.2 Excerpts A and B).
//   qkv_chain_*            the seven-launch chain the fusion replaces (same page,
//                          §2): kept as bitwise comparators.
// Every kernel except the comparators writes the fused result in one launch per
// layer, for both layer classes; in projection-only mode the rings write the raw y.
//
// All epilogue forms call the same device functions below, in the same order of
// f32 operations (explicit _rn intrinsics, no contraction), so their results
// agree bit for bit — the page's gate for the fusion (§2, "The fusion's bitwise
// legitimacy").  The rings take each pair's (cos, sin) from a table the CTA fills
// once per launch with the same sincosf of the same f32 angle.
//
// Projection design (HBM-bound: ~1 flop per weight byte against a ridge of
// ~270 flop/B): every weight byte is read from HBM once, x is staged once per CTA
// in shared memory, each lane takes a strided share of a row's 16-byte chunks, and
// the dot products are reduced with a xor-shuffle butterfly (identical result in
// every lane).  Both rows of a neox pair (j, j + hd/2) of one head are finished in
// one place, so RoPE needs no exchange between CTAs.  Each row is reduced by the
// same code whatever class the layer has, so a concat layer and the same rows split
// into wq / wk / wv give identical bits (same page, §2, "Why the concat matmul is
// bitwise").
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "epilogue_math.cuh"
#include "ptx_sync.cuh"
#include "qkv_internal.h"

namespace {
using namespace qkv_epi;
using namespace qkv_ptx;

constexpr int kUnroll = 4;  // 16-byte loads in flight per lane per row

// Device status word: [0] flags (bit 0 = position out of range), [1] a bad position.
__device__ unsigned int g_qkv_status[2];

// ---------------------------------------------------------------- PTX helpers

// 16-byte weight load: read-only for the kernel's lifetime, streamed once,
// so it bypasses L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// ---------------------------------------------------------------- status flags

constexpr unsigned int kFlagPosRange = 1u;
constexpr unsigned int kFlagTimeout = 2u;
// ---------------------------------------------------------------- epilogue math
// rope_theta, rope_rotate, kv_put, pos_ok: epilogue_math.cuh (shared with prefill).

__device__ __forceinline__ void flag_bad_pos(int pos) {
    atomicOr(&g_qkv_status[0], kFlagPosRange);
    atomicExch(&g_qkv_status[1], static_cast<unsigned int>(pos));
}

__device__ __forceinline__ void flag_timeout() { atomicOr(&g_qkv_status[0], kFlagTimeout); }

// Limit of every bounded wait of a launch: the default, unless a test shortened it.
__device__ __forceinline__ uint64_t wait_limit(const DecodeParams& p) {
    return p.wait_limit_ns ? p.wait_limit_ns : kWaitTimeoutNs;
}

// q/k pair (j, j2) after the bias: rotate by the angle whose (cos, sin) is cs, write
// back, store k rows to the cache.
__device__ __forceinline__ void epi_qk_rot_cs(const DecodeParams& p, int sec, int j, int j2, float x0, float x1,
                                              int pos, float2 cs, bool store) {
    float r0, r1;
    rope_rotate_cs(x0, x1, cs, r0, r1);
    float* o = p.out[sec];
    o[j] = r0;
    o[j2] = r1;
    if (sec == 1 && store) {
        const size_t row = static_cast<size_t>(pos) * static_cast<size_t>(p.nkt);
        kv_put(p.kv_k, p.kv_f16, row + j, r0);
        kv_put(p.kv_k, p.kv_f16, row + j2, r1);
    }
}

// The same with the angle of frequency inv_freq at pos.
__device__ __forceinline__ void epi_qk_rot(const DecodeParams& p, int sec, int j, int j2, float x0, float x1,
                                           int pos, float inv_freq, bool store) {
    epi_qk_rot_cs(p, sec, j, j2, x0, x1, pos, rope_cos_sin(pos, inv_freq), store);
}

__device__ __forceinline__ void epi_qk_pair_b(const DecodeParams& p, int sec, int j, int j2, float y0, float y1,
                                              float b0, float b1, int pos, float inv_freq, bool store) {
    epi_qk_rot(p, sec, j, j2, __fadd_rn(y0, b0), __fadd_rn(y1, b1), pos, inv_freq, store);
}

__device__ __forceinline__ void epi_qk_pair(const DecodeParams& p, int sec, int j, int j2, float y0, float y1,
                                            int pos, float inv_freq, bool store) {
    epi_qk_pair_b(p, sec, j, j2, y0, y1, p.bias[sec][j], p.bias[sec][j2], pos, inv_freq, store);
}

// v element: bias (already loaded), write back, store to the cache.
__device__ __forceinline__ void epi_v_elem_b(const DecodeParams& p, int j, float y, float b, int pos, bool store) {
    const float val = __fadd_rn(y, b);
    p.out[2][j] = val;
    if (store) kv_put(p.kv_v, p.kv_f16, static_cast<size_t>(pos) * static_cast<size_t>(p.nkt) + j, val);
}

__device__ __forceinline__ void epi_v_elem(const DecodeParams& p, int j, float y, int pos, bool store) {
    epi_v_elem_b(p, j, y, p.bias[2][j], pos, store);
}

// ---------------------------------------------------------------- projection

// Unit u -> (section, row pair, pair index d).  q and k units are the neox pairs
// (h*hd + d, h*hd + d + hd/2); v units are adjacent rows (2u', 2u' + 1).
__device__ __forceinline__ void unit_rows(int u, int qpairs, int kpairs, int half, int hd, int& sec,
                                          int& r0, int& r1, int& d) {
    if (u < qpairs + kpairs) {
        sec = (u < qpairs) ? 0 : 1;
        const int v = (u < qpairs) ? u : u - qpairs;
        const int h = v / half;
        d = v - h * half;
        r0 = h * hd + d;
        r1 = r0 + half;
    } else {
        sec = 2;
        d = 0;
        r0 = 2 * (u - qpairs - kpairs);
        r1 = r0 + 1;
    }
}

// acc += sum of 8 bf16 weights (one 16-byte chunk) times x[8c .. 8c+7].
__device__ __forceinline__ float fma_chunk_bf16(uint4 w, float4 xa, float4 xb, float acc) {
    acc = __fmaf_rn(bf16_lo(w.x), xa.x, acc);
    acc = __fmaf_rn(bf16_hi(w.x), xa.y, acc);
    acc = __fmaf_rn(bf16_lo(w.y), xa.z, acc);
    acc = __fmaf_rn(bf16_hi(w.y), xa.w, acc);
    acc = __fmaf_rn(bf16_lo(w.z), xb.x, acc);
    acc = __fmaf_rn(bf16_hi(w.z), xb.y, acc);
    acc = __fmaf_rn(bf16_lo(w.w), xb.z, acc);
    acc = __fmaf_rn(bf16_hi(w.w), xb.w, acc);
    return acc;
}

// acc += sum of 4 f32 weights times x[4c .. 4c+3].
__device__ __forceinline__ float fma_chunk_f32(uint4 w, float4 x, float acc) {
    acc = __fmaf_rn(__uint_as_float(w.x), x.x, acc);
    acc = __fmaf_rn(__uint_as_float(w.y), x.y, acc);
    acc = __fmaf_rn(__uint_as_float(w.z), x.z, acc);
    acc = __fmaf_rn(__uint_as_float(w.w), x.w, acc);
    return acc;
}

// Per-lane partial dot products of two rows with the staged x.  Lane l takes
// 16-byte chunks l, l + 32, l + 64, ... in increasing order.
//   bf16 rows: x staged as two planes of float4 (x[8c..8c+3], x[8c+4..8c+7]) so a
//              warp's shared loads are contiguous.
//   f32 rows:  x staged as float4 x[4c..4c+3].
template <typename WT>
__device__ __forceinline__ void dot2_vec(const WT* row0, const WT* row1, const float4* xs, int H,
                                         int lane, float& a0, float& a1) {
    constexpr bool kBf16 = sizeof(WT) == 2;
    constexpr int kPerChunk = kBf16 ? 8 : 4;
    const int nch = H / kPerChunk;
    const uint4* w0 = reinterpret_cast<const uint4*>(row0);
    const uint4* w1 = reinterpret_cast<const uint4*>(row1);
    const float4* xb = xs + nch;  // second plane (bf16 only)
    a0 = 0.f;
    a1 = 0.f;
    int c = lane;
    for (; c + 32 * (kUnroll - 1) < nch; c += 32 * kUnroll) {
        uint4 v0[kUnroll], v1[kUnroll];
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            v0[i] = ld_stream(w0 + c + 32 * i);
            v1[i] = ld_stream(w1 + c + 32 * i);
        }
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            const int cc = c + 32 * i;
            if constexpr (kBf16) {
                const float4 xa = xs[cc], xb2 = xb[cc];
                a0 = fma_chunk_bf16(v0[i], xa, xb2, a0);
                a1 = fma_chunk_bf16(v1[i], xa, xb2, a1);
            } else {
                const float4 xv = xs[cc];
                a0 = fma_chunk_f32(v0[i], xv, a0);
                a1 = fma_chunk_f32(v1[i], xv, a1);
            }
        }
    }
    for (; c < nch; c += 32) {
        const uint4 v0 = ld_stream(w0 + c), v1 = ld_stream(w1 + c);
        if constexpr (kBf16) {
            const float4 xa = xs[c], xb2 = xb[c];
            a0 = fma_chunk_bf16(v0, xa, xb2, a0);
            a1 = fma_chunk_bf16(v1, xa, xb2, a1);
        } else {
            const float4 xv = xs[c];
            a0 = fma_chunk_f32(v0, xv, a0);
            a1 = fma_chunk_f32(v1, xv, a1);
        }
    }
}

template <typename WT>
__device__ __forceinline__ float w_value(const WT* row, int i);
template <>
__device__ __forceinline__ float w_value<float>(const float* row, int i) {
    return __ldg(row + i);
}
template <>
__device__ __forceinline__ float w_value<uint16_t>(const uint16_t* row, int i) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(row + i)) << 16);
}

// Scalar path for rows that are not 16-byte aligned: lane l takes elements
// l, l + 32, ... in increasing order; x staged plainly.
template <typename WT>
__device__ __forceinline__ void dot2_scalar(const WT* row0, const WT* row1, const float* xs, int H,
                                            int lane, float& a0, float& a1) {
    a0 = 0.f;
    a1 = 0.f;
    for (int i = lane; i < H; i += 32) {
        const float xv = xs[i];
        a0 = __fmaf_rn(w_value(row0, i), xv, a0);
        a1 = __fmaf_rn(w_value(row1, i), xv, a1);
    }
}

// Stage x (and the frequency table) in shared memory.
// Stage the projection input x in shared memory, threads tid = 0 .. nthr-1: bf16 rows
// get two float4 planes (x[8c..8c+3] at c, x[8c+4..8c+7] at nch + c), aligned f32
// rows x in order, unaligned rows scalars.  The caller synchronises before reading.
template <typename WT, bool VEC>
__device__ __forceinline__ void stage_plain(const DecodeParams& p, float4* xs4, int tid, int nthr) {
    const int H = p.H;
    if constexpr (VEC && sizeof(WT) == 2) {
        const int nch = H / 8;
        const float4* xg = reinterpret_cast<const float4*>(p.x);
        for (int c = tid; c < nch; c += nthr) {
            xs4[c] = xg[2 * c];
            xs4[nch + c] = xg[2 * c + 1];
        }
    } else if constexpr (VEC) {
        const int nch = H / 4;
        const float4* xg = reinterpret_cast<const float4*>(p.x);
        for (int c = tid; c < nch; c += nthr) xs4[c] = xg[c];
    } else {
        float* xs = reinterpret_cast<float*>(xs4);
        for (int i = tid; i < H; i += nthr) xs[i] = p.x[i];
    }
}

// Shared partial sums of h^2, one per staging warp.
__device__ __forceinline__ float* norm_partials() {
    __shared__ float red_s[32];
    return red_s;
}

// RMSNorm(h) = (h * w) * inv with inv = 1 / sqrt(sum(h^2) / H + eps) a scalar of the
// layer, so y = W RMSNorm(h) = inv * (W (h * w)): stage x' = h * w (p.x being h and
// p.norm_w w) and, in the same pass, each warp's sum of h^2 (each thread its elements
// in order, then a warp tree); norm_inv() adds the warps in order after the caller's
// barrier, and the kernel scales each dot product by inv.  The reduction so runs beside
// the staging instead of in front of it.
template <typename WT, bool VEC>
__device__ __forceinline__ void stage_normed(const DecodeParams& p, float4* xs4, int tid, int nthr) {
    const int H = p.H;
    const float* nw = p.norm_w;
    float ss = 0.f;
    const float4* nw4 = reinterpret_cast<const float4*>(nw);  // 16-byte aligned (checked on the host)
    auto take4 = [&](float4 h, int i4) {
        const float4 w = nw4[i4];
        ss = __fmaf_rn(h.x, h.x, ss);
        ss = __fmaf_rn(h.y, h.y, ss);
        ss = __fmaf_rn(h.z, h.z, ss);
        ss = __fmaf_rn(h.w, h.w, ss);
        return make_float4(__fmul_rn(h.x, w.x), __fmul_rn(h.y, w.y), __fmul_rn(h.z, w.z), __fmul_rn(h.w, w.w));
    };
    if constexpr (VEC && sizeof(WT) == 2) {
        const int nch = H / 8;
        const float4* xg = reinterpret_cast<const float4*>(p.x);
#pragma unroll 4
        for (int c = tid; c < nch; c += nthr) {
            xs4[c] = take4(xg[2 * c], 2 * c);
            xs4[nch + c] = take4(xg[2 * c + 1], 2 * c + 1);
        }
    } else if constexpr (VEC) {
        const int nch = H / 4;
        const float4* xg = reinterpret_cast<const float4*>(p.x);
#pragma unroll 4
        for (int c = tid; c < nch; c += nthr) xs4[c] = take4(xg[c], c);
    } else {
        float* xs = reinterpret_cast<float*>(xs4);
#pragma unroll 4
        for (int i = tid; i < H; i += nthr) {
            const float h = p.x[i];
            ss = __fmaf_rn(h, h, ss);
            xs[i] = __fmul_rn(h, nw[i]);
        }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) norm_partials()[tid >> 5] = ss;
}

// The norm weight is a parameter: its lines can be brought into L1 before the
// dependency wait, so the staging after it finds them there.
__device__ __forceinline__ void prefetch_norm(const DecodeParams& p, int tid, int nthr) {
    if (p.norm_w == nullptr) return;
    for (int i = tid * 32; i < p.H; i += nthr * 32)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(p.norm_w + i));
}

// 1 / sqrt(sum(h^2) / H + eps) from the staging warps' partials (after the barrier that
// follows the staging), or 1 for a layer without a norm.
__device__ __forceinline__ float norm_inv(const DecodeParams& p, int nthr) {
    if (p.norm_w == nullptr) return 1.f;
    const float* red = norm_partials();
    float tot = red[0];
    for (int w = 1; w < nthr / 32; ++w) tot = __fadd_rn(tot, red[w]);
    return __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, static_cast<float>(p.H)), p.norm_eps)));
}

// The projection input: h * w and the partials of sum(h^2) when the layer has a norm
// weight (the kernel then scales its dot products by norm_inv), else x as given.
template <typename WT, bool VEC>
__device__ __forceinline__ void stage_input(const DecodeParams& p, float4* xs4, int tid, int nthr) {
    if (p.norm_w != nullptr)
        stage_normed<WT, VEC>(p, xs4, tid, nthr);
    else
        stage_plain<WT, VEC>(p, xs4, tid, nthr);
}

template <typename WT, bool VEC, int MODE>
__global__ void __launch_bounds__(256) qkv_decode_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ float4 smem4[];
    __shared__ float freq_s[QKV_MAX_HEAD_DIM / 2];
    const int lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    const int gwarp = blockIdx.x * wpc + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * wpc;
    const int half = p.hd >> 1;
    const int qpairs = p.nqt >> 1, kpairs = p.nkt >> 1;
    const int units = qpairs + kpairs + (p.nkt >> 1);

    // Inputs written upstream (x, pos) are read, and outputs written, only
    // after the preceding grid in the stream has completed.
    prefetch_norm(p, threadIdx.x, blockDim.x);
    griddep_wait();
    stage_input<WT, VEC>(p, smem4, threadIdx.x, blockDim.x);
    for (int i = threadIdx.x; i < (p.hd >> 1); i += blockDim.x) freq_s[i] = p.inv_freq[i];
    __syncthreads();
    const float inv = norm_inv(p, blockDim.x);
    const int pos = (MODE == kFused) ? *p.pos : 0;
    const bool store = pos_ok(pos, p.n_ctx);
    griddep_launch_dependents();
    if (MODE == kFused && !store && blockIdx.x == 0 && threadIdx.x == 0) flag_bad_pos(pos);

    for (int u = gwarp; u < units; u += nwarps) {
        int sec, r0, r1, d;
        unit_rows(u, qpairs, kpairs, half, p.hd, sec, r0, r1, d);
        const WT* w = static_cast<const WT*>(p.w[sec]);
        const size_t H = static_cast<size_t>(p.H);
        float a0, a1;
        if constexpr (VEC) dot2_vec<WT>(w + r0 * H, w + r1 * H, smem4, p.H, lane, a0, a1);
        else dot2_scalar<WT>(w + r0 * H, w + r1 * H, reinterpret_cast<const float*>(smem4), p.H, lane, a0, a1);
        a0 = warp_sum(a0);
        a1 = warp_sum(a1);
        if (p.norm_w != nullptr) {
            a0 = __fmul_rn(a0, inv);
            a1 = __fmul_rn(a1, inv);
        }
        if (lane == 0) {
            if constexpr (MODE == kProjectOnly) {
                p.out[sec][r0] = a0;
                p.out[sec][r1] = a1;
            } else if (sec < 2) {
                epi_qk_pair(p, sec, r0, r1, a0, a1, pos, freq_s[d], store);
            } else {
                epi_v_elem(p, r0, a0, pos, store);
                epi_v_elem(p, r1, a1, pos, store);
            }
        }
    }
}

// ---------------------------------------------------------------- bulk-copy pipelined projection

// Persistent variant for 16-byte aligned rows: one CTA per SM owns a
// share of the row-pair units (a contiguous range, or for rows under 4 KB units
// b, b + grid, ...).  A producer warp streams each unit's two
// rows (2 x H weights) into a ring of shared-memory stages with cp.async.bulk
// (L2 evict-first: each byte is used once), ahead of the consumers.  Consumer
// group g (G warps) owns stages g, g + NG, ... and reduces whole units from
// shared memory: with a stage count that is a multiple of the group count NG,
// unit i and unit i - S (the previous user of its stage) belong to the same
// group, so every group waits on each stage's phases strictly in order and a
// parity wait can never alias a phase two rounds ahead.  The G warps of a
// group split the 16-byte chunks of the unit's rows (thread t of the group
// takes chunks t, t + 32G, ...) and combine their partials in warp order
// through shared memory under a group-wide named barrier.  The producer starts before griddepcontrol.wait:
// weights are never written by the preceding grid, so under programmatic
// dependent launch a layer's weight stream starts while the previous layer
// finishes.
//
// Per row the sum is: group thread t takes chunks t, t + 32G, ... in
// increasing order, accumulating even and odd elements in the two halves of
// packed f32x2 FMAs; the halves are added, a xor butterfly sums each warp,
// then the G warp partials are added in warp order.  The order depends only
// on H and G, not on the layer class, so concat and mixed layers give
// identical bits.
#ifndef QKV_DECODE_GROUP_WARPS
#define QKV_DECODE_GROUP_WARPS 1
#endif
constexpr int kGroupWarps = QKV_DECODE_GROUP_WARPS;   // G: warps per group
// Launch shapes: rows of >= 8 KB (one neox pair per stage is >= 16 KB) use one
// CTA per SM with 5 consumer groups; shorter rows use two CTAs per SM with 3
// groups each, which keeps more independent producers streaming.
#ifndef QKV_DECODE_LARGE_GROUPS
#define QKV_DECODE_LARGE_GROUPS 5
#endif
#ifndef QKV_DECODE_LARGE_CTAS
#define QKV_DECODE_LARGE_CTAS 1
#endif
#ifndef QKV_DECODE_LARGE_SMEM_KB
#define QKV_DECODE_LARGE_SMEM_KB 225
#endif
#ifndef QKV_DECODE_SMALL_GROUPS
#define QKV_DECODE_SMALL_GROUPS 3
#endif
#ifndef QKV_DECODE_SMALL_CTAS
#define QKV_DECODE_SMALL_CTAS 2
#endif
#ifndef QKV_DECODE_SMALL_SMEM_KB
#define QKV_DECODE_SMALL_SMEM_KB 110
#endif
constexpr int kGroupsLarge = QKV_DECODE_LARGE_GROUPS;
constexpr int kGroupsSmall = QKV_DECODE_SMALL_GROUPS;
constexpr size_t kSmallRowBytes = 8192;
// Rows under 4 KB (the 0.5B shape's 3.5 KB f32 rows) run the pair ring three CTAs per SM
// with two groups each: more, smaller CTAs, so a layer's CTAs start while the previous
// layer's are still finishing (0.5B sweep +12 %; the 7 KB rows of the 7B shape lose with it).
constexpr int kGroupsTiny = 2;
constexpr int kTinyCtas = 3;
constexpr int kTinySmemKb = 72;
constexpr size_t kTinyRowBytes = 4096;

#ifndef QKV_DECODE_PAIRS
#define QKV_DECODE_PAIRS 1
#endif
constexpr int kPairs = QKV_DECODE_PAIRS;  // P: neox pairs per unit (rows per bulk copy)

// Unit u of the ring kernel: up to P consecutive neox pairs (d0 .. d0+n-1) of
// one q or k head — two contiguous blocks of n rows, (h*hd + d0 ...) and
// (h*hd + hd/2 + d0 ...) — or 2n consecutive v rows (blocks r.. and r+n..).
struct Unit {
    int sec;  // 0 q, 1 k, 2 v
    int r;    // first row of block A (section-local)
    int n;    // rows per block
    int off;  // block B starts at row r + off
    int d;    // q / k: pair index of row r within its head (r mod hd); v: 0
};

template <int P = kPairs>
__device__ __forceinline__ Unit unit_info(int u, int nqt, int nkt, int hd) {
    const int half = hd >> 1;
    const int per_head = (half + P - 1) / P;
    const int uq = (nqt / hd) * per_head, uk = (nkt / hd) * per_head;
    Unit t;
    if (u < uq + uk) {
        t.sec = (u < uq) ? 0 : 1;
        const int v = t.sec ? u - uq : u;
        const int h = v / per_head;
        const int d0 = (v - h * per_head) * P;
        t.n = min(P, half - d0);
        t.r = h * hd + d0;
        t.off = half;
        t.d = d0;
    } else {
        t.sec = 2;
        t.r = (u - uq - uk) * 2 * P;
        t.n = min(P, (nkt - t.r) >> 1);
        t.off = t.n;
        t.d = 0;
    }
    return t;
}

// Units of the pair ring (one neox pair per unit), decoded without a runtime division when
// hd / 2 is a power of two (every Qwen head width): the nqt / 2 q pairs, then the nkt / 2 k
// pairs, then the v row pairs.  Gives the Unit that unit_info<1> gives.
struct PairUnits {
    int uq, uk, half, shift, hd, nkt;
    __device__ __forceinline__ explicit PairUnits(const DecodeParams& p)
        : uq(p.nqt >> 1), uk(p.nkt >> 1), half(p.hd >> 1), shift(-1), hd(p.hd), nkt(p.nkt) {
        int e = 0;
        while ((1 << e) < half) ++e;
        if ((1 << e) == half) shift = e;
    }
    __device__ __forceinline__ Unit at(int u) const {
        Unit t;
        if (u < uq + uk) {
            t.sec = u < uq ? 0 : 1;
            const int v = t.sec ? u - uq : u;
            const int h = shift >= 0 ? (v >> shift) : v / half;
            t.d = v - h * half;
            t.r = h * hd + t.d;
            t.n = 1;
            t.off = half;
        } else {
            t.sec = 2;
            t.r = 2 * (u - uq - uk);
            t.n = min(1, (nkt - t.r) >> 1);
            t.off = t.n;
            t.d = 0;
        }
        return t;
    }
};

// Items of the next layer a pair-ring CTA brings into L2 after its own copies have landed.
constexpr int kNextLayerPrefetchItems = 2;

template <int P = kPairs>
__host__ __device__ __forceinline__ int unit_count(int nqt, int nkt, int hd) {
    const int per_head = ((hd >> 1) + P - 1) / P;
    return (nqt / hd) * per_head + (nkt / hd) * per_head + (nkt + 2 * P - 1) / (2 * P);
}

// The block ring decodes a CTA's first kUnitTable units once, before the dependency wait
// (they depend on the shape only), into a shared table instead of dividing by runtime
// values (heads, units per head) in every item: +1 % on the 14B graph.  (In the pair
// ring the table measured 0.6-2 % slower, so it decodes per item.)
constexpr int kUnitTable = 64;
// (sec, d) share the first word: sec in bits 0-1, d above.
__device__ __forceinline__ int4 pack_unit(const Unit& t) { return make_int4(t.sec | (t.d << 2), t.r, t.n, t.off); }
__device__ __forceinline__ Unit unpack_unit(int4 v) {
    Unit t;
    t.sec = v.x & 3;
    t.d = v.x >> 2;
    t.r = v.y;
    t.n = v.z;
    t.off = v.w;
    return t;
}

// First unit of CTA b of `grid` when `units` are split in contiguous ranges:
// units * F(b / grid) with F(x) = x + (skew / 100) x (1 - x).  CTAs of a chained
// launch are dispatched in block order as the previous grid's SMs free up, so later
// blocks start later; skew > 0 gives them proportionally less (the first block
// 1 + skew/100 times the mean share, the last 1 - skew/100) and the ranges end
// together.  skew = 0 is the even split.  Monotone for 0 <= skew <= 100.
__host__ __device__ __forceinline__ int unit_split(int units, int b, int grid, int skew) {
    const long long u = units, bb = b, g = grid;
    return static_cast<int>((u * bb * (100 * g + skew * (g - bb))) / (100 * g * g));
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ float4 ld_shared_f4(const void* p) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// acc += 16-byte weight chunk * its x slice (bf16: 8 values in xa, xb; f32: 4
// values in xa), even elements in acc.x, odd in acc.y.
template <typename WT>
__device__ __forceinline__ float2 fma2_chunk(uint4 w, float4 xa, float4 xb, float2 acc) {
    if constexpr (sizeof(WT) == 2) {
        acc = __ffma2_rn(bf16x2_to_f32x2(w.x), make_float2(xa.x, xa.y), acc);
        acc = __ffma2_rn(bf16x2_to_f32x2(w.y), make_float2(xa.z, xa.w), acc);
        acc = __ffma2_rn(bf16x2_to_f32x2(w.z), make_float2(xb.x, xb.y), acc);
        acc = __ffma2_rn(bf16x2_to_f32x2(w.w), make_float2(xb.z, xb.w), acc);
    } else {
        acc = __ffma2_rn(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), make_float2(xa.x, xa.y), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), make_float2(xa.z, xa.w), acc);
    }
    return acc;
}

// Both rows of a unit, staged: group thread t takes chunks t, t + 32G, ...; x
// is staged as float4 planes (bf16: x[8c..8c+3] and x[8c+4..8c+7]; f32:
// x[4c..4c+3]).  Returns the warp's partial of each row (same in every lane).
template <typename WT>
__device__ __forceinline__ void dot2_staged(const unsigned char* row0, const unsigned char* row1,
                                            const float4* xs, int H, int t, float& a0, float& a1) {
    constexpr bool kBf16 = sizeof(WT) == 2;
    const int nch = H / (kBf16 ? 8 : 4);
    const float4* xb = xs + nch;
    float2 c0 = make_float2(0.f, 0.f), c1 = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int c = t; c < nch; c += 32 * kGroupWarps) {
        const uint4 v0 = ld_shared_v4(row0 + 16 * c);
        const uint4 v1 = ld_shared_v4(row1 + 16 * c);
        const float4 xa = ld_shared_f4(xs + c);
        const float4 x2 = kBf16 ? ld_shared_f4(xb + c) : xa;
        c0 = fma2_chunk<WT>(v0, xa, x2, c0);
        c1 = fma2_chunk<WT>(v1, xa, x2, c1);
    }
    a0 = warp_sum(__fadd_rn(c0.x, c0.y));
    a1 = warp_sum(__fadd_rn(c1.x, c1.y));
}

// x held in registers (CPL > 0: every lane takes exactly CPL chunks of a row, i.e. the row
// has 32 * CPL chunks of 16 bytes): each consumer lane loads the x values of its chunks
// once per launch, so the dot loop reads only weights from shared memory.  That halves the
// loop's shared-memory reads and roughly doubles a warp's rate (one warp per SM
// sub-partition: 8.3 -> 16 B/clk on 7 KB rows).  CPL = 0: x stays in shared memory.
template <typename WT, int CPL>
struct XRegs {
    static constexpr int kF2 = sizeof(WT) == 2 ? 4 : 2;  // x pairs per 16-byte chunk
    float2 v[CPL > 0 ? CPL : 1][kF2];
};

template <typename WT, int CPL>
__device__ __forceinline__ void load_xregs(XRegs<WT, CPL>& xr, const float4* xs, int H, int t) {
    if constexpr (CPL > 0) {
        const int nch = H / (sizeof(WT) == 2 ? 8 : 4);
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const float4 xa = ld_shared_f4(xs + t + 32 * k);
            xr.v[k][0] = make_float2(xa.x, xa.y);
            xr.v[k][1] = make_float2(xa.z, xa.w);
            if constexpr (sizeof(WT) == 2) {
                const float4 xb = ld_shared_f4(xs + nch + t + 32 * k);
                xr.v[k][2] = make_float2(xb.x, xb.y);
                xr.v[k][3] = make_float2(xb.z, xb.w);
            }
        }
    }
}

// dot2_staged with x from registers: the same chunks in the same order and the same packed
// FMAs, so the same bits.
template <typename WT, int CPL>
__device__ __forceinline__ void dot2_xregs(const unsigned char* row0, const unsigned char* row1,
                                           const XRegs<WT, CPL>& xr, int t, float& a0, float& a1) {
    float2 c0 = make_float2(0.f, 0.f), c1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const uint4 v0 = ld_shared_v4(row0 + 16 * (t + 32 * k));
        const uint4 v1 = ld_shared_v4(row1 + 16 * (t + 32 * k));
        if constexpr (sizeof(WT) == 2) {
            c0 = __ffma2_rn(bf16x2_to_f32x2(v0.x), xr.v[k][0], c0);
            c1 = __ffma2_rn(bf16x2_to_f32x2(v1.x), xr.v[k][0], c1);
            c0 = __ffma2_rn(bf16x2_to_f32x2(v0.y), xr.v[k][1], c0);
            c1 = __ffma2_rn(bf16x2_to_f32x2(v1.y), xr.v[k][1], c1);
            c0 = __ffma2_rn(bf16x2_to_f32x2(v0.z), xr.v[k][2], c0);
            c1 = __ffma2_rn(bf16x2_to_f32x2(v1.z), xr.v[k][2], c1);
            c0 = __ffma2_rn(bf16x2_to_f32x2(v0.w), xr.v[k][3], c0);
            c1 = __ffma2_rn(bf16x2_to_f32x2(v1.w), xr.v[k][3], c1);
        } else {
            c0 = __ffma2_rn(make_float2(__uint_as_float(v0.x), __uint_as_float(v0.y)), xr.v[k][0], c0);
            c1 = __ffma2_rn(make_float2(__uint_as_float(v1.x), __uint_as_float(v1.y)), xr.v[k][0], c1);
            c0 = __ffma2_rn(make_float2(__uint_as_float(v0.z), __uint_as_float(v0.w)), xr.v[k][1], c0);
            c1 = __ffma2_rn(make_float2(__uint_as_float(v1.z), __uint_as_float(v1.w)), xr.v[k][1], c1);
        }
    }
    a0 = warp_sum(__fadd_rn(c0.x, c0.y));
    a1 = warp_sum(__fadd_rn(c1.x, c1.y));
}

// Chunks per lane of a row of H elements when they divide evenly among 32 lanes and a
// register-resident x is compiled for that count, else 0.
template <typename WT>
__host__ __device__ __forceinline__ int chunks_per_lane(int H) {
    const int per = sizeof(WT) == 2 ? 8 : 4;
    if (H % per != 0 || (H / per) % 32 != 0) return 0;
    return H / per / 32;
}

template <typename WT, int MODE, int kGroups, int CPL>
__global__ void __launch_bounds__((kGroups * kGroupWarps + 1) * 32, 2)
    qkv_decode_tma_kernel(const __grid_constant__ DecodeParams p, int stages, uint32_t stage_bytes,
                          uint32_t x_bytes, int skew) {
    static_assert(CPL == 0 || kGroupWarps == 1, "register-resident x needs one-warp groups");
    constexpr int kConsumerWarps = kGroups * kGroupWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float2 cs_s[QKV_MAX_HEAD_DIM / 2];  // (cos, sin) of each pair index at pos
    __shared__ float gpart[kGroups][kGroupWarps][2];
    float4* xs4 = reinterpret_cast<float4*>(smem);
    unsigned char* ring = smem + x_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(stages) * stage_bytes);
    uint64_t* empty = full + stages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = p.hd >> 1;
    const int units = unit_count(p.nqt, p.nkt, p.hd);
    // Rows under 4 KB (three CTAs per SM) take units b, b + grid, ... (0.5B sweep +2 %); the
    // 4-8 KB rows keep skewed contiguous shares (strided measured -2 % on the 7B graph).
    constexpr bool kStrided = kGroups == kGroupsTiny;
    const int u_step = kStrided ? static_cast<int>(gridDim.x) : 1;
    const int u_begin = kStrided ? static_cast<int>(blockIdx.x) : unit_split(units, blockIdx.x, gridDim.x, skew);
    const int n = kStrided ? (units > u_begin ? (units - 1 - u_begin) / static_cast<int>(gridDim.x) + 1 : 0)
                           : unit_split(units, blockIdx.x + 1, gridDim.x, skew) - u_begin;
    const uint32_t row_bytes = static_cast<uint32_t>(p.H) * sizeof(WT);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    // The next layer's grid may be scheduled now: it reads and writes nothing of
    // ours before its own griddepcontrol.wait, which waits for this grid to finish.
    griddep_launch_dependents();

    static_assert(kPairs == 1, "the pair ring decodes one neox pair per unit");
    const PairUnits pu(p);
    if (warp == kConsumerWarps) {
        // ---- producer: one lane issues all bulk copies of this CTA ----
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const uint64_t limit = wait_limit(p);
            const int n_issue = p.withhold_last_copy ? n - 1 : n;
            int issued = 0;
            for (int i = 0; i < n_issue; ++i) {
                const int s = i % stages;
                if (i >= stages && !mbar_wait_bounded(&empty[s], ((i / stages) - 1) & 1, limit)) {
                    flag_timeout();
                    break;
                }
                const Unit t = pu.at(u_begin + i * u_step);
                const unsigned char* w = static_cast<const unsigned char*>(p.w[t.sec]);
                unsigned char* dst = ring + static_cast<size_t>(s) * stage_bytes;
                const uint32_t blk = static_cast<uint32_t>(t.n) * row_bytes;
                mbar_arrive_expect_tx(&full[s], 2 * blk);
                bulk_g2s(dst, w + static_cast<size_t>(t.r) * row_bytes, blk, &full[s], pol);
                bulk_g2s(dst + blk, w + static_cast<size_t>(t.r + t.off) * row_bytes, blk, &full[s], pol);
                ++issued;
            }
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            const int first = issued > stages ? issued - stages : 0;
            for (int i = first; i < issued; ++i)
                if (!mbar_wait_bounded(&full[i % stages], (i / stages) & 1, limit)) flag_timeout();
            // In a model graph, the next layer's CTA with this index owns the same units (same
            // shape): bring its first items into L2 now, while this CTA's consumers finish and
            // the SM changes hands, so its first copies are L2 hits (7B graph +8 %).
            if (p.next_w[0] != nullptr) {
                const int npf = n < kNextLayerPrefetchItems ? n : kNextLayerPrefetchItems;
                for (int i = 0; i < npf; ++i) {
                    const Unit t = pu.at(u_begin + i * u_step);
                    const unsigned char* w = static_cast<const unsigned char*>(p.next_w[t.sec]);
                    const uint32_t blk = static_cast<uint32_t>(t.n) * row_bytes;
                    bulk_prefetch_l2(w + static_cast<size_t>(t.r) * row_bytes, blk);
                    bulk_prefetch_l2(w + static_cast<size_t>(t.r + t.off) * row_bytes, blk);
                }
            }
        }
        return;
    }

    // ---- consumers ----
    const uint64_t limit = wait_limit(p);
    prefetch_norm(p, threadIdx.x, kConsumerWarps * 32);
    griddep_wait();
    const int pos = (MODE == kFused) ? *p.pos : 0;
    {
        // Every head rotates pair d by the same angle: its (cos, sin) are computed once here.
        const int tid = threadIdx.x, nthr = kConsumerWarps * 32;
        stage_input<WT, true>(p, xs4, tid, nthr);
        if (MODE == kFused)
            for (int i = tid; i < half; i += nthr) cs_s[i] = rope_cos_sin(pos, p.inv_freq[i]);
    }
    named_barrier_sync(1, kConsumerWarps * 32);
    const float inv = norm_inv(p, kConsumerWarps * 32);
    const bool store = pos_ok(pos, p.n_ctx);
    if (MODE == kFused && !store && blockIdx.x == 0 && threadIdx.x == 0) flag_bad_pos(pos);
    XRegs<WT, CPL> xr;
    load_xregs<WT, CPL>(xr, xs4, p.H, lane);

    const int group = warp / kGroupWarps, gw = warp % kGroupWarps;
    const int gt = gw * 32 + lane;  // thread index within the group
    for (int i = group; i < n; i += kGroups) {
        const int s = i % stages;
        if (!mbar_wait_bounded(&full[s], (i / stages) & 1, limit)) {
            if (lane == 0) flag_timeout();
            break;
        }
        const Unit t = pu.at(u_begin + i * u_step);
        const unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
        const uint32_t blk = static_cast<uint32_t>(t.n) * row_bytes;
        for (int j = 0; j < t.n; ++j) {
            const int r0 = t.r + j, r1 = t.r + t.off + j;
            // the epilogue's bias loads are issued now and land during the dot product
            float b0 = 0.f, b1 = 0.f;
            if (MODE == kFused && gw == 0 && lane == 0) {
                b0 = __ldg(p.bias[t.sec] + r0);
                b1 = __ldg(p.bias[t.sec] + r1);
            }
            float a0, a1;
            if constexpr (CPL > 0) dot2_xregs<WT, CPL>(st + j * row_bytes, st + blk + j * row_bytes, xr, lane, a0, a1);
            else dot2_staged<WT>(st + j * row_bytes, st + blk + j * row_bytes, xs4, p.H, gt, a0, a1);
            const bool last = (j == t.n - 1);
            if constexpr (kGroupWarps > 1) {
                if (lane == 0) {
                    gpart[group][gw][0] = a0;
                    gpart[group][gw][1] = a1;
                }
                // the group's reads of this pair are done and its partials published
                named_barrier_sync(2 + group, 32 * kGroupWarps);
                if (gw == 0) {
                    a0 = gpart[group][0][0];
                    a1 = gpart[group][0][1];
                    for (int w = 1; w < kGroupWarps; ++w) {
                        a0 = __fadd_rn(a0, gpart[group][w][0]);
                        a1 = __fadd_rn(a1, gpart[group][w][1]);
                    }
                }
                // keep the partial slots until warp 0 of the group has read them
                named_barrier_sync(2 + kGroups + group, 32 * kGroupWarps);
            } else {
                __syncwarp();
            }
            if (last && gw == 0 && lane == 0) mbar_arrive(&empty[s]);
            if (gw == 0 && lane == 0) {
                if (p.norm_w != nullptr) {
                    a0 = __fmul_rn(a0, inv);
                    a1 = __fmul_rn(a1, inv);
                }
                if constexpr (MODE == kProjectOnly) {
                    p.out[t.sec][r0] = a0;
                    p.out[t.sec][r1] = a1;
                } else if (t.sec < 2) {
                    epi_qk_rot_cs(p, t.sec, r0, r1, __fadd_rn(a0, b0), __fadd_rn(a1, b1), pos, cs_s[t.d + j],
                                  store);
                } else {
                    epi_v_elem_b(p, r0, a0, b0, pos, store);
                    epi_v_elem_b(p, r1, a1, b1, pos, store);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- block ring

#ifndef QKV_DECODE_BLOCK_PAIRS
#define QKV_DECODE_BLOCK_PAIRS 2
#endif
constexpr int kBlkPairs = QKV_DECODE_BLOCK_PAIRS;  // rows per stage (one contiguous bulk copy)

// What the block ring computes after the projection.
enum BlockEpilogue {
    kEpiQkv = 0,      // bias, neox RoPE on q/k, KV-cache store (units: neox pairs of a head, v rows)
    kEpiSwiglu = 1,   // silu(gate) * up (units: rows i of the gate half with rows nf + i)
    kEpiQkvNorm = 2,  // as kEpiQkv with each q / k head RMS-normalised before its rotation
};

template <int EPI>
__device__ __forceinline__ int blk_unit_count(const DecodeParams& p) {
    if constexpr (EPI != kEpiSwiglu) return unit_count<kBlkPairs>(p.nqt, p.nkt, p.hd);
    else return (p.nf + kBlkPairs - 1) / kBlkPairs;
}

template <int EPI>
__device__ __forceinline__ Unit blk_unit(int u, const DecodeParams& p) {
    if constexpr (EPI != kEpiSwiglu) {
        return unit_info<kBlkPairs>(u, p.nqt, p.nkt, p.hd);
    } else {
        Unit t;
        t.sec = 0;
        t.d = 0;
        t.r = u * kBlkPairs;
        t.n = min(kBlkPairs, p.nf - t.r);
        t.off = p.nf;
        return t;
    }
}

// SwiGLU of one (gate, up) pair, each step rounded to f32: silu(g) = g / (1 + e^-g).
__device__ __forceinline__ float swiglu(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// FusedQkvNorm: finish head hh (q heads first, then k heads) whose biased values
// z = y + b sit in the output section, written by the CTAs that computed its rows.  One
// warp: sum of z^2 (lane l takes elements l, l + 32, ... in order, then a xor butterfly),
// inv = 1 / sqrt(sum / hd + eps), then pair d (lane-strided) becomes
// (z_d inv w_d, z_{d+hd/2} inv w_{d+hd/2}), rotated and stored as in the plain stage.
// The values are read at L2 (ld.global.cg): other SMs wrote them.
__device__ __forceinline__ void qknorm_finish_head(const DecodeParams& p, int hh, int pos, bool store,
                                                   const float2* cs_s, int lane) {
    const int hd = p.hd, half = hd >> 1;
    const int nhq = p.nqt / hd;
    const int sec = hh < nhq ? 0 : 1;
    const int base = (sec ? hh - nhq : hh) * hd;
    const float* z = p.out[sec] + base;
    const float* w = p.qk_norm_w[sec];
    float ss = 0.f;
    for (int i = lane; i < hd; i += 32) {
        const float v = __ldcg(z + i);
        ss = __fmaf_rn(v, v, ss);
    }
    ss = warp_sum(ss);
    const float inv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(hd)), p.qk_eps)));
    for (int d = lane; d < half; d += 32) {
        const float n0 = __fmul_rn(__fmul_rn(__ldcg(z + d), inv), __ldg(w + d));
        const float n1 = __fmul_rn(__fmul_rn(__ldcg(z + d + half), inv), __ldg(w + d + half));
        epi_qk_rot_cs(p, sec, base + d, base + d + half, n0, n1, pos, cs_s[d], store);
    }
}

// Block ring: a unit of kBlkPairs neox pairs has two row blocks, (h*hd + d0 ..)
// and (h*hd + hd/2 + d0 ..); each block is one stage, filled by one contiguous
// bulk copy.  Item i of a CTA is block (i & 1) of its local unit i >> 1 (see below
// for which units a CTA takes).  Consumer groups (one warp each) own stages g, g + NG, ...
// The consumer of a q/k block publishes its biased dot products in shared
// memory and bumps the unit's counter; the second of the two blocks to finish
// rotates the unit's pairs and stores them, one pair per lane.  v blocks need
// no partner and finish on their own.  Each row is reduced exactly as in the
// pair ring (dot2_staged), so both kernels give the same bits.  With
// EPI = kEpiSwiglu the same ring runs the FusedFFN: a unit pairs gate rows
// (i ..) with up rows (nf + i ..), and the second block writes silu(g) * u.
// Except with kEpiQkvNorm (whose heads must end up in few CTAs) a CTA takes units
// b, b + grid, b + 2 grid, ... rather than a contiguous share: in a chained launch
// the CTAs that start last (the highest block indices) then hold the smaller
// shares, and every QKV CTA ends on v rows (14B graph +1.6 %, FFN +1 %).
template <typename WT, int MODE, int kGroups, int EPI, int CPL>
__global__ void __launch_bounds__((kGroups + 1) * 32, 1)
    qkv_decode_blk_kernel(const __grid_constant__ DecodeParams p, int stages, uint32_t stage_bytes,
                          uint32_t x_bytes, int max_units, int skew) {
    static_assert(kBlkPairs >= 1 && kBlkPairs <= 8, "rows per block");
    static_assert(kGroupWarps == 1, "one warp per consumer group");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float2 cs_s[QKV_MAX_HEAD_DIM / 2];  // (cos, sin) of each pair index at pos
    __shared__ int4 unit_s[kUnitTable];              // this CTA's first units, decoded
    float4* xs4 = reinterpret_cast<float4*>(smem);
    unsigned char* ring = smem + x_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(stages) * stage_bytes);
    uint64_t* empty = full + stages;
    float* bias_s = reinterpret_cast<float*>(empty + stages);            // [max_units][2][kBlkPairs]
    float* res = bias_s + max_units * 2 * kBlkPairs;                     // [max_units][2][kBlkPairs]
    int* cnt = reinterpret_cast<int*>(res + max_units * 2 * kBlkPairs);  // [max_units]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool kStrided = EPI != kEpiQkvNorm;
    const int units = blk_unit_count<EPI>(p);
    const int b = static_cast<int>(blockIdx.x), g = static_cast<int>(gridDim.x);
    const int u_begin = kStrided ? b : unit_split(units, b, g, skew);
    const int u_step = kStrided ? g : 1;  // unit of local index ul: u_begin + ul * u_step
    const int u_end = kStrided ? 0 : unit_split(units, b + 1, g, skew);  // contiguous shares only
    const int n_units = kStrided ? (units > b ? (units - 1 - b) / g + 1 : 0) : u_end - u_begin;
    const int n = 2 * n_units;
    const uint32_t row_bytes = static_cast<uint32_t>(p.H) * sizeof(WT);

    if (threadIdx.x == 0) {
        for (int st = 0; st < stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], 1);
        }
        mbar_fence_init();
    }
    for (int i = threadIdx.x; i < max_units; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    // The next layer's grid may be scheduled now: it reads and writes nothing of
    // ours before its own griddepcontrol.wait, which waits for this grid to finish.
    griddep_launch_dependents();

    if (warp == kGroups) {
        // ---- producer: one lane issues all bulk copies of this CTA ----
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const uint64_t limit = wait_limit(p);
            const int n_issue = p.withhold_last_copy ? n - 1 : n;
            int issued = 0;
            for (int i = 0; i < n_issue; ++i) {
                const int st = i % stages;
                if (i >= stages && !mbar_wait_bounded(&empty[st], ((i / stages) - 1) & 1, limit)) {
                    flag_timeout();
                    break;
                }
                const Unit t = blk_unit<EPI>(u_begin + (i >> 1) * u_step, p);
                const int rb = (i & 1) ? t.r + t.off : t.r;
                const uint32_t bytes = static_cast<uint32_t>(t.n) * row_bytes;
                const unsigned char* w = static_cast<const unsigned char*>(p.w[t.sec]);
                mbar_arrive_expect_tx(&full[st], bytes);
                bulk_g2s(ring + static_cast<size_t>(st) * stage_bytes, w + static_cast<size_t>(rb) * row_bytes,
                         bytes, &full[st], pol);
                ++issued;
            }
            // Drain: no copy may still be landing in shared memory when the CTA exits.
            const int first = issued > stages ? issued - stages : 0;
            for (int i = first; i < issued; ++i)
                if (!mbar_wait_bounded(&full[i % stages], (i / stages) & 1, limit)) flag_timeout();
        }
        return;
    }

    // ---- consumers ----
    const uint64_t limit = wait_limit(p);
    // Biases are parameters, not outputs of an earlier kernel: stage this CTA's
    // share before the dependency wait, so no global load sits in the item loop.
    if (MODE == kFused && EPI != kEpiSwiglu) {
        const int nb = n_units * 2 * kBlkPairs;
        for (int e = threadIdx.x; e < nb; e += kGroups * 32) {
            const int j = e % kBlkPairs, blk = (e / kBlkPairs) & 1, ul = e / (2 * kBlkPairs);
            const Unit t = blk_unit<EPI>(u_begin + ul * u_step, p);
            bias_s[e] = j < t.n ? __ldg(p.bias[t.sec] + (blk ? t.r + t.off : t.r) + j) : 0.f;
        }
    }
    for (int ul = threadIdx.x; 2 * ul < n && ul < kUnitTable; ul += kGroups * 32)
        unit_s[ul] = pack_unit(blk_unit<EPI>(u_begin + ul * u_step, p));
    prefetch_norm(p, threadIdx.x, kGroups * 32);
    griddep_wait();
    const int pos = (MODE == kFused && EPI != kEpiSwiglu) ? *p.pos : 0;
    {
        // Every head rotates pair d by the same angle: its (cos, sin) are computed once here.
        const int tid = threadIdx.x, nthr = kGroups * 32;
        stage_input<WT, true>(p, xs4, tid, nthr);
        if (MODE == kFused && EPI != kEpiSwiglu)
            for (int i = tid; i < (p.hd >> 1); i += nthr) cs_s[i] = rope_cos_sin(pos, p.inv_freq[i]);
    }
    named_barrier_sync(1, kGroups * 32);
    const float inv = norm_inv(p, kGroups * 32);
    const bool store = pos_ok(pos, p.n_ctx);
    if (MODE == kFused && EPI != kEpiSwiglu && !store && blockIdx.x == 0 && threadIdx.x == 0) flag_bad_pos(pos);
    XRegs<WT, CPL> xr;
    load_xregs<WT, CPL>(xr, xs4, p.H, lane);

    for (int i = warp; i < n; i += kGroups) {
        const int st = i % stages;
        if (!mbar_wait_bounded(&full[st], (i / stages) & 1, limit)) {
            if (lane == 0) flag_timeout();
            break;
        }
        const int ul = i >> 1, blk = i & 1;
        const Unit t = ul < kUnitTable ? unpack_unit(unit_s[ul]) : blk_unit<EPI>(u_begin + ul * u_step, p);
        const int rb = blk ? t.r + t.off : t.r;
        const unsigned char* sp = ring + static_cast<size_t>(st) * stage_bytes;
        float y[kBlkPairs];
#pragma unroll
        for (int j = 0; j < kBlkPairs; j += 2) {
            // rows rb + j and rb + j + 1 (the second repeats the first past the block's end)
            const int j1 = (j + 1 < t.n) ? j + 1 : j;
            float a0 = 0.f, a1 = 0.f;
            if (j < t.n) {
                if constexpr (CPL > 0) dot2_xregs<WT, CPL>(sp + j * row_bytes, sp + j1 * row_bytes, xr, lane, a0, a1);
                else dot2_staged<WT>(sp + j * row_bytes, sp + j1 * row_bytes, xs4, p.H, lane, a0, a1);
            }
            y[j] = a0;
            if (j + 1 < kBlkPairs) y[j + 1] = a1;
        }
        if (p.norm_w != nullptr) {
#pragma unroll
            for (int j = 0; j < kBlkPairs; ++j) y[j] = __fmul_rn(y[j], inv);
        }
        __syncwarp();  // every lane is done reading the stage
        if (lane == 0) mbar_arrive(&empty[st]);
        // Epilogue: lane j < t.n takes row rb + j of the block.
        float yl = y[0];
#pragma unroll
        for (int j = 1; j < kBlkPairs; ++j)
            if (lane == j) yl = y[j];
        const int e = (ul * 2 + blk) * kBlkPairs + lane;
        if constexpr (EPI == kEpiSwiglu) {
            if (lane < t.n) res[e] = yl;
            __syncwarp();
            int first = 0;
            if (lane == 0) {
                __threadfence_block();
                first = atomicAdd(&cnt[ul], 1);
                __threadfence_block();
            }
            first = __shfl_sync(0xffffffffu, first, 0);
            __syncwarp();
            if (first == 1 && lane < t.n) {
                // the partner block is complete: gate from block 0, up from block 1
                const float o = static_cast<volatile float*>(res)[e + (blk ? -kBlkPairs : kBlkPairs)];
                p.out[0][t.r + lane] = swiglu(blk ? o : yl, blk ? yl : o);
            }
        } else if constexpr (MODE == kProjectOnly) {
            if (lane < t.n) p.out[t.sec][rb + lane] = yl;
        } else if (t.sec == 2) {
            if (lane < t.n) epi_v_elem_b(p, rb + lane, yl, bias_s[e], pos, store);
        } else if constexpr (EPI == kEpiQkvNorm) {
            // a head's norm needs all of its rows: publish z = y + b; the head's last CTA finishes it
            if (lane < t.n) p.out[t.sec][rb + lane] = __fadd_rn(yl, bias_s[e]);
        } else {
            const float yb = lane < t.n ? __fadd_rn(yl, bias_s[e]) : 0.f;
            if (lane < t.n) res[e] = yb;
            __syncwarp();
            int first = 0;
            if (lane == 0) {
                __threadfence_block();
                first = atomicAdd(&cnt[ul], 1);
                __threadfence_block();
            }
            first = __shfl_sync(0xffffffffu, first, 0);
            __syncwarp();
            if (first == 1 && lane < t.n) {
                // the partner block is complete: rotate the unit's pair lane
                const float o = static_cast<volatile float*>(res)[e + (blk ? -kBlkPairs : kBlkPairs)];
                const int r0 = t.r + lane;
                epi_qk_rot_cs(p, t.sec, r0, r0 + t.off, blk ? o : yb, blk ? yb : o, pos, cs_s[t.d + lane], store);
            }
        }
    }
    if constexpr (EPI == kEpiQkvNorm && MODE == kFused) {
        // Every raw q / k value of this CTA is written; count this CTA's units into each
        // head it touched.  The CTA that completes a head's count finishes that head.
        named_barrier_sync(1, kGroups * 32);
        const int per_head = ((p.hd >> 1) + kBlkPairs - 1) / kBlkPairs;
        const int qk_end = min(u_end, (p.nqt / p.hd + p.nkt / p.hd) * per_head);
        if (u_begin < qk_end) {
            const int h0 = u_begin / per_head, h1 = (qk_end - 1) / per_head;
            for (int hh = h0 + warp; hh <= h1; hh += kGroups) {
                const int mine = min(qk_end, (hh + 1) * per_head) - max(u_begin, hh * per_head);
                int last = 0;
                if (lane == 0) {
                    // One acquire-release count: the release publishes this CTA's values of head
                    // hh (every consumer warp wrote its values before the barrier above), the
                    // acquire makes the other contributors' values visible to the CTA that
                    // completes the count (in place of fence, atomic, fence: +2.6 % on 14B).
                    unsigned int old;
                    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                                 : "=r"(old)
                                 : "l"(&p.head_cnt[hh]), "r"(static_cast<unsigned int>(mine))
                                 : "memory");
                    last = old + mine == static_cast<unsigned int>(per_head);
                    if (last) p.head_cnt[hh] = 0u;  // every contributor has counted: ready for the next launch
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                // A shuffle does not order memory: the barrier orders every lane's reads of
                // the other CTAs' values after lane 0's acquiring fence.
                __syncwarp();
                if (last) qknorm_finish_head(p, hh, pos, store, cs_s, lane);
            }
        }
    }
}

// ---------------------------------------------------------------- standalone epilogue

// One thread per unit of the flat index: q pairs, then k pairs, then v elements.
__global__ void __launch_bounds__(256) qkv_epilogue_kernel(const __grid_constant__ DecodeParams p) {
    __shared__ float freq_s[QKV_MAX_HEAD_DIM / 2];
    for (int i = threadIdx.x; i < (p.hd >> 1); i += blockDim.x) freq_s[i] = p.inv_freq[i];
    griddep_wait();
    __syncthreads();
    const int half = p.hd >> 1;
    const int qpairs = p.nqt >> 1, kpairs = p.nkt >> 1;
    const int total = qpairs + kpairs + p.nkt;
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    const int pos = *p.pos;
    const bool store = pos_ok(pos, p.n_ctx);
    if (!store && u == 0) flag_bad_pos(pos);
    if (u >= total) return;
    if (u < qpairs + kpairs) {
        const int sec = (u < qpairs) ? 0 : 1;
        const int v = (u < qpairs) ? u : u - qpairs;
        const int h = v / half;
        const int d = v - h * half;
        const int j = h * p.hd + d, j2 = j + half;
        const float* io = p.out[sec];
        epi_qk_pair(p, sec, j, j2, io[j], io[j2], pos, freq_s[d], store);
    } else {
        const int j = u - qpairs - kpairs;
        epi_v_elem(p, j, p.out[2][j], pos, store);
    }
}

// ---------------------------------------------------------------- unfused chain

__global__ void qkv_chain_add_bias_kernel(float* y, const float* b, int64_t n) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) y[i] = __fadd_rn(y[i], b[i]);
}

__global__ void qkv_chain_rope_kernel(const __grid_constant__ DecodeParams p, float* y, int n_heads) {
    const int half = p.hd >> 1;
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= n_heads * half) return;
    const int h = u / half, d = u - h * half;
    const int j = h * p.hd + d, j2 = j + half;
    const int pos = *p.pos;
    float r0, r1;
    rope_rotate(y[j], y[j2], rope_theta(pos, p.inv_freq[d]), r0, r1);
    y[j] = r0;
    y[j2] = r1;
}

__global__ void qkv_chain_store_kernel(const __grid_constant__ DecodeParams p, const float* src, void* cache) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    const int pos = *p.pos;
    const bool store = pos_ok(pos, p.n_ctx);
    if (!store && j == 0) flag_bad_pos(pos);
    if (j >= p.nkt || !store) return;
    kv_put(cache, p.kv_f16, static_cast<size_t>(pos) * static_cast<size_t>(p.nkt) + j, src[j]);
}

// ---------------------------------------------------------------- launch helpers

template <typename K>
cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t stream,
                      const DecodeParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    }
    return n;
}

// Dynamic shared memory per CTA: the ring takes what one CTA per SM can have,
// which keeps the most weight bytes in flight.
#ifndef QKV_DECODE_MAX_STAGES
#define QKV_DECODE_MAX_STAGES 32
#endif
constexpr int kMaxStages = QKV_DECODE_MAX_STAGES;
// Work skew (percent) of the ring kernels in a chained launch: see unit_split.  The
// pair ring (rows of 4-8 KB: 7B-size layers, 8 us each) gains from it (+4 % at 20 on the
// 7B graph); the block ring's 12-unit shares are too coarse to skew without imbalance
// (the FusedQkvNorm ring keeps even contiguous shares; the others take strided units).
#ifndef QKV_DECODE_CHAIN_SKEW_PAIR
#define QKV_DECODE_CHAIN_SKEW_PAIR 20
#endif
#ifndef QKV_DECODE_CHAIN_SKEW_BLOCK
#define QKV_DECODE_CHAIN_SKEW_BLOCK 0
#endif
constexpr int kChainSkewPair = QKV_DECODE_CHAIN_SKEW_PAIR;
constexpr int kChainSkewBlock = QKV_DECODE_CHAIN_SKEW_BLOCK;

struct RingShape {
    int stages;        // multiple of the group count
    int ctas_per_sm;
    uint32_t stage_bytes, x_bytes;
};

// Ring for this layer in a dynamic shared-memory budget, or stages = 0 when the
// shape needs the register-streaming kernel (unaligned rows, or rows too long to
// stage).
template <typename WT>
RingShape ring_shape(const DecodeParams& p, int groups, int ctas_per_sm, int smem_kb) {
    RingShape r = {};
    const size_t row = static_cast<size_t>(p.H) * sizeof(WT);
    const size_t budget = static_cast<size_t>(smem_kb) * 1024;
    r.ctas_per_sm = ctas_per_sm;
    r.stage_bytes = static_cast<uint32_t>((2 * kPairs * row + 127) / 128 * 128);
    r.x_bytes = static_cast<uint32_t>((static_cast<size_t>(p.H) * 4 + 127) / 128 * 128);
    const size_t barriers = 2 * 32 * sizeof(uint64_t);
    if (r.x_bytes + barriers + static_cast<size_t>(groups) * r.stage_bytes > budget) return r;
    int st = static_cast<int>((budget - r.x_bytes - barriers) / r.stage_bytes);
    st = st > kMaxStages ? kMaxStages : st;
    st -= st % groups;
    r.stages = st;
    return r;
}

template <typename WT, int MODE, int kGroups, int CPL = 0>
cudaError_t launch_decode_tma(const DecodeParams& p, const RingShape& r, bool pdl, cudaStream_t stream) {
    auto kernel = qkv_decode_tma_kernel<WT, MODE, kGroups, CPL>;
    const size_t smem = r.x_bytes + static_cast<size_t>(r.stages) * r.stage_bytes + 2 * r.stages * sizeof(uint64_t);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int units = unit_count(p.nqt, p.nkt, p.hd);
    const int ctas = sm_count() * r.ctas_per_sm;
    const int grid = units < ctas ? units : ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((kGroups * kGroupWarps + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    // a skew needs a few units per CTA to move; below that it only unbalances
    const int skew = (pdl && units >= 4 * grid) ? kChainSkewPair : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p, r.stages, r.stage_bytes, r.x_bytes, skew);
}


// Block ring in a dynamic shared-memory budget (0 stages: does not fit).
template <typename WT, int MODE, int kGroups, int EPI = kEpiQkv, int CPL = 0>
cudaError_t launch_decode_blk(const DecodeParams& p, int ctas_per_sm, int smem_kb, bool pdl, cudaStream_t stream,
                              bool& launched) {
    launched = false;
    const size_t row = static_cast<size_t>(p.H) * sizeof(WT);
    const uint32_t stage_bytes = static_cast<uint32_t>((kBlkPairs * row + 127) / 128 * 128);
    const uint32_t x_bytes = static_cast<uint32_t>((static_cast<size_t>(p.H) * 4 + 127) / 128 * 128);
    const int units =
        EPI != kEpiSwiglu ? unit_count<kBlkPairs>(p.nqt, p.nkt, p.hd) : (p.nf + kBlkPairs - 1) / kBlkPairs;
    const int ctas_max = sm_count() * ctas_per_sm;
    const int grid = units < ctas_max ? units : ctas_max;
    const int skew = pdl ? kChainSkewBlock : 0;
    int max_units = 0;
    if (EPI != kEpiQkvNorm) {
        max_units = (units + grid - 1) / grid;  // units b, b + grid, ...
    } else {
        for (int b = 0; b < grid; ++b) {
            const int nb = unit_split(units, b + 1, grid, skew) - unit_split(units, b, grid, skew);
            max_units = nb > max_units ? nb : max_units;
        }
    }
    // per unit: staged biases, published results and a counter
    const size_t tail = static_cast<size_t>(max_units) * (4 * kBlkPairs * sizeof(float) + sizeof(int));
    const size_t budget = static_cast<size_t>(smem_kb) * 1024;
    const size_t fixed = x_bytes + tail + 2 * 32 * sizeof(uint64_t);
    if (fixed + static_cast<size_t>(kGroups) * stage_bytes > budget) return cudaSuccess;
    int stages = static_cast<int>((budget - fixed) / stage_bytes);
    stages = stages > kMaxStages ? kMaxStages : stages;
    stages -= stages % kGroups;
    auto kernel = qkv_decode_blk_kernel<WT, MODE, kGroups, EPI, CPL>;
    const size_t smem = x_bytes + static_cast<size_t>(stages) * stage_bytes + 2 * stages * sizeof(uint64_t) + tail;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((kGroups + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    launched = true;
    return cudaLaunchKernelEx(&cfg, kernel, p, stages, stage_bytes, x_bytes, max_units, skew);
}

// Register-resident x is compiled for the row widths of the Qwen2.5 workloads (chunks per
// lane 20: H 5120 bf16; 14: H 3584 bf16; 7: H 896 f32) in fused launches; every other
// width, and projection-only launches, keep x in shared memory (same bits either way).
template <typename WT, int MODE, int kGroups, int EPI>
cudaError_t launch_blk_any(const DecodeParams& p, int ctas_per_sm, int smem_kb, bool pdl, cudaStream_t stream,
                           bool& launched) {
    if constexpr (MODE == kFused) {
        const int cpl = chunks_per_lane<WT>(p.H);
        if constexpr (sizeof(WT) == 2 && kGroups == kGroupsLarge) {
            if (cpl == 20) return launch_decode_blk<WT, MODE, kGroups, EPI, 20>(p, ctas_per_sm, smem_kb, pdl, stream, launched);
        }
        if constexpr (sizeof(WT) == 2 && kGroups == kGroupsSmall && EPI == kEpiSwiglu) {
            if (cpl == 14) return launch_decode_blk<WT, MODE, kGroups, EPI, 14>(p, ctas_per_sm, smem_kb, pdl, stream, launched);
        }
        if constexpr (sizeof(WT) == 4 && kGroups == kGroupsSmall && EPI == kEpiSwiglu) {
            if (cpl == 7) return launch_decode_blk<WT, MODE, kGroups, EPI, 7>(p, ctas_per_sm, smem_kb, pdl, stream, launched);
        }
    }
    return launch_decode_blk<WT, MODE, kGroups, EPI, 0>(p, ctas_per_sm, smem_kb, pdl, stream, launched);
}

template <typename WT, int MODE, int kGroups>
cudaError_t launch_tma_any(const DecodeParams& p, const RingShape& r, bool pdl, cudaStream_t stream) {
    if constexpr (MODE == kFused) {
        const int cpl = chunks_per_lane<WT>(p.H);
        if constexpr (sizeof(WT) == 2 && kGroups == kGroupsSmall) {
            if (cpl == 14) return launch_decode_tma<WT, MODE, kGroups, 14>(p, r, pdl, stream);
        }
        if constexpr (sizeof(WT) == 4 && kGroups == kGroupsTiny) {
            if (cpl == 7) return launch_decode_tma<WT, MODE, kGroups, 7>(p, r, pdl, stream);
        }
    }
    return launch_decode_tma<WT, MODE, kGroups, 0>(p, r, pdl, stream);
}

template <typename WT, bool VEC, int MODE>
cudaError_t launch_decode_t(const DecodeParams& p, bool pdl, cudaStream_t stream) {
    if constexpr (VEC) {
        const size_t row = static_cast<size_t>(p.H) * sizeof(WT);
        if (row >= kSmallRowBytes) {
            // rows of >= 8 KB: block ring (one contiguous copy per stage), else the pair ring
            bool launched = false;
            const cudaError_t e = launch_blk_any<WT, MODE, kGroupsLarge, kEpiQkv>(p, QKV_DECODE_LARGE_CTAS,
                                                                                   QKV_DECODE_LARGE_SMEM_KB, pdl,
                                                                                   stream, launched);
            if (launched || e != cudaSuccess) return e;
            const RingShape r = ring_shape<WT>(p, kGroupsLarge, QKV_DECODE_LARGE_CTAS, QKV_DECODE_LARGE_SMEM_KB);
            if (r.stages > 0) return launch_decode_tma<WT, MODE, kGroupsLarge>(p, r, pdl, stream);
        } else if (row < kTinyRowBytes) {
            const RingShape r = ring_shape<WT>(p, kGroupsTiny, kTinyCtas, kTinySmemKb);
            if (r.stages > 0) return launch_tma_any<WT, MODE, kGroupsTiny>(p, r, pdl, stream);
        } else {
            const RingShape r = ring_shape<WT>(p, kGroupsSmall, QKV_DECODE_SMALL_CTAS, QKV_DECODE_SMALL_SMEM_KB);
            if (r.stages > 0) return launch_tma_any<WT, MODE, kGroupsSmall>(p, r, pdl, stream);
        }
    }
    auto kernel = qkv_decode_kernel<WT, VEC, MODE>;
    const size_t smem = static_cast<size_t>(p.H) * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    const int units = (p.nqt >> 1) + (p.nkt >> 1) + (p.nkt >> 1);
    // Small layers: 4-warp CTAs spread the rows over more SMs.
    const int wpc = (units >= 8 * 152) ? 8 : 4;
    const int grid = (units + wpc - 1) / wpc;
    return launch_ex(kernel, dim3(grid), dim3(wpc * 32), smem, pdl, stream, p);
}

template <typename WT>
cudaError_t launch_ffn_t(const DecodeParams& p, bool pdl, cudaStream_t stream) {
    const size_t row = static_cast<size_t>(p.H) * sizeof(WT);
    bool launched = false;
    const cudaError_t e =
        row >= kSmallRowBytes
            ? launch_blk_any<WT, kFused, kGroupsLarge, kEpiSwiglu>(p, QKV_DECODE_LARGE_CTAS, QKV_DECODE_LARGE_SMEM_KB,
                                                                  pdl, stream, launched)
            : launch_blk_any<WT, kFused, kGroupsSmall, kEpiSwiglu>(p, QKV_DECODE_SMALL_CTAS, QKV_DECODE_SMALL_SMEM_KB,
                                                                  pdl, stream, launched);
    if (e != cudaSuccess) return e;
    return launched ? cudaSuccess : cudaErrorNotSupported;
}

template <typename WT>
cudaError_t launch_qknorm_t(const DecodeParams& p, bool pdl, cudaStream_t stream) {
    const size_t row = static_cast<size_t>(p.H) * sizeof(WT);
    bool launched = false;
    const cudaError_t e =
        row >= kSmallRowBytes
            ? launch_blk_any<WT, kFused, kGroupsLarge, kEpiQkvNorm>(p, QKV_DECODE_LARGE_CTAS,
                                                                   QKV_DECODE_LARGE_SMEM_KB, pdl, stream, launched)
            : launch_blk_any<WT, kFused, kGroupsSmall, kEpiQkvNorm>(p, QKV_DECODE_SMALL_CTAS,
                                                                   QKV_DECODE_SMALL_SMEM_KB, pdl, stream, launched);
    if (e != cudaSuccess) return e;
    return launched ? cudaSuccess : cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_qknorm(const DecodeParams& p, int w_dtype, bool pdl, cudaStream_t stream) {
    return w_dtype == QKV_BF16 ? launch_qknorm_t<uint16_t>(p, pdl, stream) : launch_qknorm_t<float>(p, pdl, stream);
}

// Library-owned per-head counters for callers that cannot allocate device memory: a
// fixed array in the module's global memory, present on every device that loads the
// library, holding kQknormStaticHeads counters (4 KB).
static __device__ __align__(256) unsigned int g_qknorm_static_counters[kQknormStaticHeads];

// Id of the context current on this thread (0 when none is), through the driver entry
// points the runtime exposes (no link against the driver library).
static unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

cudaError_t qknorm_static_workspace(unsigned int** out) {
    // Host code cannot use the array's name as a device address: look the address up
    // with the device current, once per device and context, and reuse it.  The context
    // id keys the cache, so after cudaDeviceReset (which unloads the module; the next
    // call runs in a new primary context) the address is looked up again.
    static std::mutex mu;
    static unsigned int* addr[kQknormMaxDevices] = {};
    static unsigned long long ctx_of[kQknormMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kQknormMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_qknorm_static_counters);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<unsigned int*>(p);
        ctx_of[dev] = current_context_id();  // the lookup made the device's context current
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_ffn(const DecodeParams& p, int w_dtype, bool pdl, cudaStream_t stream) {
    return w_dtype == QKV_BF16 ? launch_ffn_t<uint16_t>(p, pdl, stream) : launch_ffn_t<float>(p, pdl, stream);
}

cudaError_t launch_decode(const DecodeParams& p, int w_dtype, int vec, DecodeMode mode, bool pdl,
                          cudaStream_t stream) {
    if (w_dtype == QKV_BF16) {
        if (vec) return mode == kFused ? launch_decode_t<uint16_t, true, kFused>(p, pdl, stream)
                                       : launch_decode_t<uint16_t, true, kProjectOnly>(p, pdl, stream);
        return mode == kFused ? launch_decode_t<uint16_t, false, kFused>(p, pdl, stream)
                              : launch_decode_t<uint16_t, false, kProjectOnly>(p, pdl, stream);
    }
    if (vec) return mode == kFused ? launch_decode_t<float, true, kFused>(p, pdl, stream)
                                   : launch_decode_t<float, true, kProjectOnly>(p, pdl, stream);
    return mode == kFused ? launch_decode_t<float, false, kFused>(p, pdl, stream)
                          : launch_decode_t<float, false, kProjectOnly>(p, pdl, stream);
}

cudaError_t launch_epilogue(const DecodeParams& p, cudaStream_t stream) {
    const int total = (p.nqt >> 1) + (p.nkt >> 1) + p.nkt;
    const int grid = (total + 255) / 256;
    return launch_ex(qkv_epilogue_kernel, dim3(grid), dim3(256), 0, false, stream, p);
}

cudaError_t launch_chain_add_bias(float* y, const float* b, int64_t n, cudaStream_t stream) {
    const int64_t grid = (n + 255) / 256;
    qkv_chain_add_bias_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(y, b, n);
    return cudaGetLastError();
}

cudaError_t launch_chain_rope(const DecodeParams& p, float* y, int n_heads, cudaStream_t stream) {
    const int total = n_heads * (p.hd >> 1);
    qkv_chain_rope_kernel<<<(total + 255) / 256, 256, 0, stream>>>(p, y, n_heads);
    return cudaGetLastError();
}

cudaError_t launch_chain_store(const DecodeParams& p, const float* src, void* cache, cudaStream_t stream) {
    qkv_chain_store_kernel<<<(p.nkt + 255) / 256, 256, 0, stream>>>(p, src, cache);
    return cudaGetLastError();
}

cudaError_t device_status_read(cudaStream_t stream, uint32_t* flags, int32_t* bad_pos) {
    unsigned int h[2] = {0u, 0u};
    cudaError_t e = cudaMemcpyFromSymbolAsync(h, g_qkv_status, sizeof(h), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (h[0] != 0u) {
        const unsigned int zero[2] = {0u, 0u};
        e = cudaMemcpyToSymbolAsync(g_qkv_status, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return e;
    }
    *flags = h[0];
    *bad_pos = static_cast<int32_t>(h[1]);
    return cudaSuccess;
}
