// Prefill (nt >= 1 tokens) of the attention-input stage on sm_103a: the dense
// contraction Y = X W^T on the 5th-generation tensor cores, with the per-token
// epilogue (bias, neox RoPE at positions[t], KV-cache store) applied to the
// accumulator as it leaves tensor memory.
//
// The page keeps prefill on the unfused chain (its fused epilogue is gated to
// nt == 1: "73 · D3-8 — G4 FusedQKV ported to CUDA", §3.2 Excerpt D and §3.3);
// the per-token math is the decode math of §3.2 Excerpt A at pos = positions[t],
// computed by the same device functions (epilogue_math.cuh).
//
// Tiling.  A pair tile is 128 tokens (UMMA M) x 64 weight rows: two 32-row
// boxes chosen so that every neox pair lands in one thread — for a q or k tile
// rows (h*hd + d0 .. +31) and (h*hd + hd/2 + d0 .. +31), for a v tile 64
// consecutive rows.  A thread-block cluster of S CTAs owns S consecutive pair
// tiles and splits K (64-wide blocks, 128 bytes: one 128B-swizzle row) into S
// ranges: each CTA multiplies its K range of X by the W rows of all S tiles
// (one UMMA with N = 64 S), so it stages 1/S of X per weight row.  Warp 0 lane 0
// streams W boxes into its ring, warp 2 lane 0 the X blocks into another (mbarrier
// transaction counts), both after the dependency wait; warp 1 lane 0 issues
// tcgen05.mma (kind::f16, bf16 x bf16 -> f32 in TMEM, K = 16 per instruction) and
// frees stages with tcgen05.commit.  After
// the K loop each CTA hands its partial sums of every other tile to that tile's
// CTA through distributed shared memory (staged locally and sent as one bulk
// copy, counted in bytes on the receiver's mbarrier), and CTA r adds the S
// partials of tile r in rank order, so the result does not depend on which CTA
// finishes first.  All four warps then run the epilogue of tile r, one token per thread:
// bias, RoPE (its (cos, sin) computed while the K loop runs), Y through shared
// memory (128-byte swizzle) and two TMA tensor stores, the token's k/v cache
// rows as 16-byte stores.  Every wait is bounded; on expiry the kernel flags the
// device status word, drains in-flight copies and MMAs, frees TMEM and returns.
// Once the exchange is over no CTA touches a peer's shared memory, so the CTAs
// of a cluster leave independently.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "epilogue_math.cuh"
#include "ptx_sync.cuh"
#include "qkv_internal.h"

namespace {
using namespace qkv_epi;
using namespace qkv_ptx;

constexpr int kBM = 128;                       // tokens per tile (UMMA M)
constexpr int kBN = 64;                        // weight rows per tile (UMMA N)
constexpr int kBox = 32;                       // rows per W box
constexpr int kBK = 64;                        // K per stage (bf16): 128 bytes
constexpr int kUK = 16;                        // K per tcgen05.mma, kind::f16
// The epilogue splits each tile's 32 neox pairs in kParts column parts: warps w and
// w + 4k read the same TMEM lanes (tokens), each its own part, so the per-token work
// of a thread shrinks kParts-fold; the extra warps idle through the K loop.
#ifndef QKV_PREFILL_EPI_PARTS
#define QKV_PREFILL_EPI_PARTS 4
#endif
constexpr int kParts = QKV_PREFILL_EPI_PARTS;
static_assert(kParts == 1 || kParts == 2 || kParts == 4, "column parts");
constexpr int kThreads = 128 * kParts;
constexpr uint32_t kABlk = kBM * kBK * 2;      // 16 KB: one X block (128 tokens x 64 K)
constexpr uint32_t kTileBlk = kBN * kBK * 2;   // 8 KB: one pair tile's W block (64 rows x 64 K)
constexpr uint32_t kBoxBytes = kBox * kBK * 2; // 4 KB
constexpr size_t kRingBytes = 224 * 1024;      // X ring + W ring
constexpr uint32_t kXchgStride = kBN + 4;      // floats per token row of an exchange slot (padded)
constexpr uint32_t kXchgSlot = kBM * kXchgStride * 4;

// Shape of a cluster of S CTAs.  The cluster owns S consecutive pair tiles
// (64 weight rows each) and splits K in S ranges; every CTA multiplies its K
// range of X by the S tiles' W rows (UMMA N = 64 S) and ends with partial sums
// of all S tiles.  kSub 64-wide K blocks form a stage.
template <int S>
struct Split {
    static_assert(S == 1 || S == 2, "clusters of 1 or 2 CTAs");
    static constexpr int kN = kBN * S;                        // UMMA N and TMEM columns
    static constexpr int kSub = 2;
    static constexpr uint32_t kXStage = kSub * kABlk;
    static constexpr uint32_t kWBlk = S * kTileBlk;           // W bytes of one K block
    static constexpr uint32_t kWStage = kSub * kWBlk;
    static constexpr int kXStages = S == 1 ? 4 : 3;
    static constexpr int kWStages = static_cast<int>((kRingBytes - kXStages * kXStage) / kWStage);
    static constexpr size_t kSmem = 1024 /* alignment slack */ + kXStages * kXStage + kWStages * kWStage +
                                    (2 * kXStages + 2 * kWStages + 4) * sizeof(uint64_t) + 16;
    static_assert(kXStages * kXStage + kWStages * kWStage <= kRingBytes, "rings");
    static_assert(kSmem <= 227 * 1024, "prefill rings exceed shared memory");
    // after the K loop the rings hold S exchange slots and the Y staging boxes
    static_assert(S * kXchgSlot + 2 * kBM * kBox * 4 <= kRingBytes, "exchange space");
    // instruction descriptor, kind::f16: D f32, A and B bf16, both K-major
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                       (static_cast<uint32_t>(kN >> 3) << 17) | ((kBM >> 4) << 24);
};

constexpr unsigned int kFlagPosRange = 1u;
constexpr unsigned int kFlagTimeout = 2u;

// Device status word of the prefill kernels: [0] flags, [1] a bad position.
__device__ unsigned int g_prefill_status[2];

__device__ __forceinline__ void flag_bad_pos(int pos) {
    atomicOr(&g_prefill_status[0], kFlagPosRange);
    atomicExch(&g_prefill_status[1], static_cast<unsigned int>(pos));
}
__device__ __forceinline__ void flag_timeout() { atomicOr(&g_prefill_status[0], kFlagTimeout); }

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Shared -> global tensor store of one box (rows past the tensor's extent are
// not written); completion tracked by this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

// Commit this thread's bulk stores and wait until their shared-memory sources
// have been read (the global writes complete on their own before the grid does).
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of `p`'s offset in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Remote arrive (release, cluster scope) on an mbarrier at a shared::cluster address.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Bounded wait with cluster-scope acquire (the arrival came from a peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Bulk copy of `bytes` from this CTA's shared memory to a peer's (shared::cluster address),
// completion counted in bytes on the peer's mbarrier.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                               uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_cluster),
                 "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster)
                 : "memory");
}

// All threads of every CTA in the cluster; release/acquire orders shared-memory
// state (barrier initialisation) across the cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked
// along M/N (stride-dimension byte offset 1024), descriptor version 1,
// layout type SWIZZLE_128B (2).  The leading-dimension offset is unused for
// swizzled K-major operands and set to 1 (16 bytes).
__device__ __forceinline__ uint64_t smem_desc_k128(const void* tile) {
    const uint64_t addr = smem_u32(tile);
    uint64_t d = 0;
    d |= (addr & 0x3FFFFull) >> 4;        // bits 0-13: start address >> 4
    d |= 1ull << 16;                      // bits 16-29: leading byte offset >> 4
    d |= (1024ull >> 4) << 32;            // bits 32-45: stride byte offset >> 4
    d |= 1ull << 46;                      // bits 46-48: fixed 0b001
    d |= 2ull << 61;                      // bits 61-63: 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 consecutive f32 columns of this warp's 32 TMEM lanes: thread l gets lane
// (warp's base lane + l), columns col .. col + 31.
__device__ __forceinline__ void tc_ld_32cols(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 / 8 consecutive f32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tc_ld_16cols(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_ld_8cols(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// N (8, 16 or 32) consecutive columns.
template <int N>
__device__ __forceinline__ void tc_ld_cols(uint32_t taddr, float* v) {
    if constexpr (N == 32) tc_ld_32cols(taddr, v);
    else if constexpr (N == 16) tc_ld_16cols(taddr, v);
    else tc_ld_8cols(taddr, v);
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- kernel

// Section and section-local first rows of pair tile `tile` (64 weight rows): for
// a q or k tile the boxes (h*hd + d0 ..) and (h*hd + hd/2 + d0 ..), for a v tile
// 64 consecutive rows.  `base` is the section's first global row.
struct PairTile {
    int sec, rowA, rowB, d0, base;
};

__device__ __forceinline__ PairTile pair_tile(int tile, const PrefillParams& p) {
    PairTile t;
    const int half = p.hd >> 1;
    const int tiles_per_head = p.hd / kBN;
    const int tq = p.nqt / kBN, tk = p.nkt / kBN;
    if (tile < tq + tk) {
        t.sec = tile < tq ? 0 : 1;
        const int v = t.sec ? tile - tq : tile;
        const int h = v / tiles_per_head;
        t.d0 = (v - h * tiles_per_head) * kBox;
        t.rowA = h * p.hd + t.d0;
        t.rowB = t.rowA + half;
    } else {
        t.sec = 2;
        t.d0 = 0;
        t.rowA = (tile - tq - tk) * kBN;
        t.rowB = t.rowA + kBox;
    }
    t.base = t.sec == 0 ? 0 : (t.sec == 1 ? p.nqt : p.nqt + p.nkt);
    return t;
}

// TMEM column of the first accumulator of box A / box B of cluster tile q.  With one W box
// per cluster (BLOCK: the cluster's tiles are 128 consecutive weight rows, loaded as one
// 16 KB box per K block in row order), a q/k head of 128 rows holds tile 0 in columns 0-31
// and 64-95 and tile 1 in 32-63 and 96-127 (the neox partner of row d is d + 64); a head of
// 64 rows, and the v rows, are tile-contiguous as with one box per 32 rows.
template <bool BLOCK>
__device__ __forceinline__ uint32_t tile_col_a(int q, int sec, int hd) {
    return (BLOCK && sec < 2 && hd == 128) ? static_cast<uint32_t>(q * kBox) : static_cast<uint32_t>(q * kBN);
}
template <bool BLOCK>
__device__ __forceinline__ uint32_t tile_col_b(int q, int sec, int hd) {
    return (BLOCK && sec < 2 && hd == 128) ? static_cast<uint32_t>(hd / 2 + q * kBox)
                                           : static_cast<uint32_t>(q * kBN + kBox);
}

template <int S, bool BLOCK>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ PrefillParams p) {
    static_assert(!BLOCK || S == 2, "one W box per cluster covers two pair tiles");
    using C = Split<S>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ float bias_s[kBN];
    __shared__ float freq_s[kBox];
    __shared__ uint32_t tmem_slot;
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sA = smem;                              // X ring
    unsigned char* sB = smem + C::kXStages * C::kXStage;   // W ring
    uint64_t* xfull = reinterpret_cast<uint64_t*>(sB + C::kWStages * C::kWStage);
    uint64_t* xempty = xfull + C::kXStages;
    uint64_t* wfull = xempty + C::kXStages;
    uint64_t* wempty = wfull + C::kWStages;
    uint64_t* done = wempty + C::kWStages;
    uint64_t* xb = done + 1;  // exchange: [0] peer idle, [1] peer's copy in, [2] own copy landed

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kBM;
    const uint64_t limit = p.wait_limit_ns ? p.wait_limit_ns : kWaitTimeoutNs;
    const uint32_t rank = S > 1 ? cluster_rank() : 0u;
    // this CTA's K range, in 64-wide blocks, and the pair tiles of its cluster
    const int nkb = (p.H + kBK - 1) / kBK;
    const int kb_lo = static_cast<int>(rank) * nkb / S, kb_hi = (static_cast<int>(rank) + 1) * nkb / S;
    const int n_stages = (kb_hi - kb_lo + C::kSub - 1) / C::kSub;
    const int tile0 = (blockIdx.x / S) * S;  // first pair tile of the cluster
    const PairTile own = pair_tile(tile0 + static_cast<int>(rank), p);  // the tile this CTA finishes

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_slot)),
                     "r"(static_cast<uint32_t>(C::kN))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < C::kXStages; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 1);
        }
        for (int s = 0; s < C::kWStages; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], 1);
        }
        mbar_init(done, 1);
        mbar_init(&xb[0], 1);
        mbar_init(&xb[1], 1);
        mbar_init(&xb[2], 1);
        mbar_fence_init();
        if (S == 2) mbar_arrive_expect_tx(&xb[1], kXchgSlot);
    }
    if (threadIdx.x < kBox) bias_s[threadIdx.x] = p.bias[own.base + own.rowA + threadIdx.x];
    else if (threadIdx.x < 2 * kBox) bias_s[threadIdx.x] = p.bias[own.base + own.rowB + threadIdx.x - kBox];
    else if (threadIdx.x < 3 * kBox && own.sec < 2) freq_s[threadIdx.x - 2 * kBox] = p.inv_freq[own.d0 + threadIdx.x - 2 * kBox];
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // The next grid may be scheduled now (it waits for this one before it reads
    // anything this one writes).  X, positions and the outputs may belong to the
    // preceding grid in the stream: every thread waits for it before touching them.
    // The W stream waits too, although weights are parameters: the next layer's CTAs
    // that land on SMs this layer leaves idle start when this layer starts, and their
    // W copies issued at once (a dedicated producer warp that does not wait) compete
    // with this layer's first stages and cost 3 % per layer.
    griddep_launch_dependents();
    griddep_wait();

    if (warp == 0 && lane == 0) {
        // ---- W producer: per K block, the two 32-row boxes of each of the S pair tiles ----
        prefetch_tensormap(&tm_w);
        {
            // Warm L2 with this cluster's share of the X rows in this CTA's K range: every
            // cluster reads each X block at about the same time, so its first reads would
            // otherwise wait for HBM together.
            const int k_lo = kb_lo * kBK, k_n = min(kb_hi * kBK, p.H) - k_lo;
            const int ncl = static_cast<int>(gridDim.x) / S, cl = static_cast<int>(blockIdx.x) / S;
            for (int t = m0 + cl; t < min(m0 + kBM, p.nt); t += ncl)
                bulk_prefetch_l2(p.X + static_cast<size_t>(t) * p.H + k_lo, static_cast<uint32_t>(k_n) * 2u);
        }
        int issued = 0;
        for (int st = 0; st < n_stages; ++st) {
            const int s = st % C::kWStages;
            if (st >= C::kWStages && !mbar_wait_bounded(&wempty[s], ((st / C::kWStages) - 1) & 1, limit)) {
                flag_timeout();
                break;
            }
            const int kb0 = kb_lo + st * C::kSub;
            const int valid = min(C::kSub, kb_hi - kb0);
            mbar_arrive_expect_tx(&wfull[s], static_cast<uint32_t>(valid) * C::kWBlk);
            for (int j = 0; j < valid; ++j) {
                const int kc = (kb0 + j) * kBK;
                if constexpr (BLOCK) {
                    // the cluster's two tiles are 128 consecutive rows from the first tile's box A
                    const PairTile pt = pair_tile(tile0, p);
                    tma_load_2d(sB + s * C::kWStage + j * C::kWBlk, &tm_w, kc, pt.base + pt.rowA, &wfull[s]);
                } else {
#pragma unroll
                    for (int t = 0; t < S; ++t) {
                        const PairTile pt = pair_tile(tile0 + t, p);
                        unsigned char* b = sB + s * C::kWStage + j * C::kWBlk + t * kTileBlk;
                        tma_load_2d(b, &tm_w, kc, pt.base + pt.rowA, &wfull[s]);
                        tma_load_2d(b + kBoxBytes, &tm_w, kc, pt.base + pt.rowB, &wfull[s]);
                    }
                }
            }
            ++issued;
        }
        // Drain: every W copy has landed and the MMAs released the last stages.
        const int first = issued > C::kWStages ? issued - C::kWStages : 0;
        for (int st = first; st < issued; ++st) {
            if (!mbar_wait_bounded(&wfull[st % C::kWStages], (st / C::kWStages) & 1, limit)) flag_timeout();
            if (!mbar_wait_bounded(&wempty[st % C::kWStages], (st / C::kWStages) & 1, limit)) flag_timeout();
        }
    } else if (warp == 2 && lane == 0) {
        // ---- X producer: 128 x 64 X blocks of this CTA's K range ----
        prefetch_tensormap(&tm_x);
        int issued = 0;
        for (int st = 0; st < n_stages; ++st) {
            const int s = st % C::kXStages;
            if (st >= C::kXStages && !mbar_wait_bounded(&xempty[s], ((st / C::kXStages) - 1) & 1, limit)) {
                flag_timeout();
                break;
            }
            const int kb0 = kb_lo + st * C::kSub;
            const int valid = min(C::kSub, kb_hi - kb0);
            mbar_arrive_expect_tx(&xfull[s], static_cast<uint32_t>(valid) * kABlk);
            for (int j = 0; j < valid; ++j)
                tma_load_2d(sA + s * C::kXStage + j * kABlk, &tm_x, (kb0 + j) * kBK, m0, &xfull[s]);
            ++issued;
        }
        const int first = issued > C::kXStages ? issued - C::kXStages : 0;
        for (int st = first; st < issued; ++st) {
            if (!mbar_wait_bounded(&xfull[st % C::kXStages], (st / C::kXStages) & 1, limit)) flag_timeout();
            if (!mbar_wait_bounded(&xempty[st % C::kXStages], (st / C::kXStages) & 1, limit)) flag_timeout();
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: D[128 x 64 S] += X block * (S tiles' W block)^T ----
        for (int st = 0; st < n_stages; ++st) {
            const int xs = st % C::kXStages, ws = st % C::kWStages;
            if (!mbar_wait_bounded(&xfull[xs], (st / C::kXStages) & 1, limit) ||
                !mbar_wait_bounded(&wfull[ws], (st / C::kWStages) & 1, limit)) {
                flag_timeout();
                break;
            }
            tc_fence_after();
            const int valid = min(C::kSub, kb_hi - (kb_lo + st * C::kSub));
            for (int j = 0; j < valid; ++j) {
                const unsigned char* a = sA + xs * C::kXStage + j * kABlk;
                const unsigned char* b = sB + ws * C::kWStage + j * C::kWBlk;
#pragma unroll
                for (int k = 0; k < kBK / kUK; ++k)
                    tc_mma(tmem, smem_desc_k128(a + k * kUK * 2), smem_desc_k128(b + k * kUK * 2), C::kIdesc,
                           (st | j | k) != 0);
            }
            tc_commit(&wempty[ws]);  // both stages are free once these MMAs have read them
            tc_commit(&xempty[xs]);
        }
        tc_commit(done);  // arrives when every MMA issued above has completed
    }

    // ---- partial sums: thread (warp, lane) owns TMEM lane 32*(warp%4) + lane = token m0 + that,
    // and pairs c0 .. c0 + kPc - 1 of the tile (columns c0.. of box A and 32 + c0.. of box B) ----
    constexpr int kPc = kBox / kParts;
    const int quarter = warp & 3;
    const int c0 = (warp >> 2) * kPc;
    const int tl = quarter * 32 + lane;  // this thread's token within the tile
    const int t = m0 + tl;
    // The token's position and the (cos, sin) of this thread's pairs, while the K loop runs
    // (the three lanes with a role above compute theirs after it).
    const int pos = t < p.nt ? p.positions[t] : 0;
    float2 cs[kPc];
    if (own.sec < 2) {
#pragma unroll
        for (int i = 0; i < kPc; ++i) cs[i] = rope_cos_sin(pos, freq_s[c0 + i]);
    }
    __syncwarp();
    // Warp-uniform: tcgen05.ld below is a warp-collective instruction.
    const bool acc_ready = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(done, 0, limit));
    if (!acc_ready && lane == 0) flag_timeout();
    tc_fence_after();
    const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* xchg = reinterpret_cast<float*>(smem);  // S slots of [128 tokens x kXchgStride], after the K loop
    float aa[kPc], ab[kPc];  // this thread's pairs: box A and box B values
    bool ready = acc_ready;  // the accumulator and, for S == 2, the peer's partial are in
    if constexpr (S == 2) {
        const uint32_t q = rank ^ 1u;
        float* mine = xchg + rank * kBM * kXchgStride;  // this CTA's partial of tile q, staged locally
        if (acc_ready) {
            float va[kPc], vb[kPc];
            tc_ld_cols<kPc>(taddr + tile_col_a<BLOCK>(static_cast<int>(q), own.sec, p.hd) + c0, va);
            tc_ld_cols<kPc>(taddr + tile_col_b<BLOCK>(static_cast<int>(q), own.sec, p.hd) + c0, vb);
            tc_ld_cols<kPc>(taddr + tile_col_a<BLOCK>(static_cast<int>(rank), own.sec, p.hd) + c0, aa);
            tc_ld_cols<kPc>(taddr + tile_col_b<BLOCK>(static_cast<int>(rank), own.sec, p.hd) + c0, ab);
            tc_wait_ld();
            float* d = mine + tl * kXchgStride;
#pragma unroll
            for (int c = 0; c < kPc; c += 4) {
                *reinterpret_cast<float4*>(d + c0 + c) = make_float4(va[c], va[c + 1], va[c + 2], va[c + 3]);
                *reinterpret_cast<float4*>(d + kBox + c0 + c) = make_float4(vb[c], vb[c + 1], vb[c + 2], vb[c + 3]);
            }
        }
        fence_proxy_async_smem();  // the staged partial is read by the bulk copy
        __syncthreads();
        if (threadIdx.x == 0) {
            // This CTA's rings are idle: the peer may copy into slot q here.
            mbar_arrive_remote(map_to_rank(&xb[0], q));
            if (!mbar_wait_cluster_bounded(&xb[0], 0, limit))
                flag_timeout();
            else if (!p.withhold_xchg)
                bulk_s2cluster(map_to_rank(mine, q), mine, kXchgSlot, map_to_rank(&xb[1], q));
        }
        // The peer's partial of this CTA's tile, in slot q (the copy's bytes complete xb[1]).
        // Without it the tile is not written.
        const bool got = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&xb[1], 0, limit));
        if (!got && lane == 0) flag_timeout();
        ready = ready && got;
        if (threadIdx.x == 0) mbar_arrive_remote(map_to_rank(&xb[2], q));  // the peer's copy has landed
    }
    if (ready) {
        if constexpr (S == 1) {
            tc_ld_cols<kPc>(taddr + tile_col_a<BLOCK>(static_cast<int>(rank), own.sec, p.hd) + c0, aa);
            tc_ld_cols<kPc>(taddr + tile_col_b<BLOCK>(static_cast<int>(rank), own.sec, p.hd) + c0, ab);
            tc_wait_ld();
        }
        if constexpr (S > 1) {
            // Sum the S K ranges in rank order (the same order in every CTA).
            float sa[kPc], sb[kPc];
            const float* s0 = xchg + tl * kXchgStride;
#pragma unroll
            for (int c = 0; c < kPc; ++c) {
                sa[c] = rank == 0 ? aa[c] : s0[c0 + c];
                sb[c] = rank == 0 ? ab[c] : s0[kBox + c0 + c];
            }
#pragma unroll 1
            for (int q = 1; q < S; ++q) {
                const float* sq = xchg + (q * kBM + tl) * kXchgStride;
                const bool mine = q == static_cast<int>(rank);
#pragma unroll
                for (int c = 0; c < kPc; ++c) {
                    sa[c] = __fadd_rn(sa[c], mine ? aa[c] : sq[c0 + c]);
                    sb[c] = __fadd_rn(sb[c], mine ? ab[c] : sq[kBox + c0 + c]);
                }
            }
#pragma unroll
            for (int c = 0; c < kPc; ++c) {
                aa[c] = sa[c];
                ab[c] = sb[c];
            }
        }
    }

    // ---- epilogue of this CTA's tile ----
    float* ys = xchg + S * (kXchgSlot / 4);  // Y staging, past the exchange slots
    if (ready) {
        const bool live = t < p.nt;
        const bool store = live && pos_ok(pos, p.n_ctx);
        if (live && !store && c0 == 0) flag_bad_pos(pos);
        if (own.sec < 2) {
#pragma unroll
            for (int i = 0; i < kPc; ++i) {
                const float x0 = __fadd_rn(aa[i], bias_s[c0 + i]);
                const float x1 = __fadd_rn(ab[i], bias_s[kBox + c0 + i]);
                float r0, r1;
                rope_rotate_cs(x0, x1, cs[i], r0, r1);
                aa[i] = r0;
                ab[i] = r1;
            }
        } else {
#pragma unroll
            for (int i = 0; i < kPc; ++i) {
                aa[i] = __fadd_rn(aa[i], bias_s[c0 + i]);
                ab[i] = __fadd_rn(ab[i], bias_s[kBox + c0 + i]);
            }
        }
        // Y: stage this thread's 16-byte chunks of row tl of both 32-column boxes, in the
        // 128-byte-swizzled layout the Y tensor map stores from.
#pragma unroll
        for (int c = 0; c < kPc / 4; ++c) {
            const int sw = (((c0 >> 2) + c) ^ (tl & 7)) * 4;
            *reinterpret_cast<float4*>(ys + tl * kBox + sw) = make_float4(aa[4 * c], aa[4 * c + 1], aa[4 * c + 2], aa[4 * c + 3]);
            *reinterpret_cast<float4*>(ys + kBM * kBox + tl * kBox + sw) =
                make_float4(ab[4 * c], ab[4 * c + 1], ab[4 * c + 2], ab[4 * c + 3]);
        }
        // k and v rows of the cache: 16-byte stores of this thread's runs of the token's row.
        if (store && own.sec > 0) {
            const size_t kvrow = static_cast<size_t>(pos) * static_cast<size_t>(p.nkt);
            void* kv = own.sec == 1 ? p.kv_k : p.kv_v;
            if (p.kv_f16) {
                __half* dst = static_cast<__half*>(kv) + kvrow;
#pragma unroll
                for (int c = 0; c < kPc / 8; ++c) {
                    uint4 ua, ub;
                    uint32_t* pa = &ua.x;
                    uint32_t* pb = &ub.x;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pa[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(aa[8 * c + 2 * e]))) |
                                (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(aa[8 * c + 2 * e + 1]))) << 16);
                        pb[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(ab[8 * c + 2 * e]))) |
                                (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(ab[8 * c + 2 * e + 1]))) << 16);
                    }
                    *reinterpret_cast<uint4*>(dst + own.rowA + c0 + 8 * c) = ua;
                    *reinterpret_cast<uint4*>(dst + own.rowB + c0 + 8 * c) = ub;
                }
            } else {
                float* dst = static_cast<float*>(kv) + kvrow;
#pragma unroll
                for (int c = 0; c < kPc / 4; ++c) {
                    *reinterpret_cast<float4*>(dst + own.rowA + c0 + 4 * c) =
                        make_float4(aa[4 * c], aa[4 * c + 1], aa[4 * c + 2], aa[4 * c + 3]);
                    *reinterpret_cast<float4*>(dst + own.rowB + c0 + 4 * c) =
                        make_float4(ab[4 * c], ab[4 * c + 1], ab[4 * c + 2], ab[4 * c + 3]);
                }
            }
        }
    }
    fence_proxy_async_smem();
    // Every warp has staged its rows (or the accumulator never became ready).
    const bool tile_ready = __syncthreads_and(ready) != 0;
    if (tile_ready && threadIdx.x == 0) {
        tma_store_2d(&tm_y, ys, own.base + own.rowA, m0);
        tma_store_2d(&tm_y, ys + kBM * kBox, own.base + own.rowB, m0);
        bulk_commit_and_wait_read();  // the boxes are read out before the CTA lets go of its shared memory
    }
    // Once the exchange is over no CTA reads or writes a peer's shared memory, so the CTAs of a
    // cluster leave independently (S == 2: after the peer reports that this CTA's copy landed,
    // so the staged source outlives the copy); the barrier orders the TMEM reads before the dealloc.
    if (S == 2 && threadIdx.x == 0 && !mbar_wait_cluster_bounded(&xb[2], 0, limit)) flag_timeout();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // After a timeout, give in-flight MMAs a second bounded wait before the
        // accumulator columns are released.
        if (!acc_ready) mbar_wait_bounded(done, 0, limit);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(static_cast<uint32_t>(C::kN))
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 2-D f32 tensor map over a row-major [rows x cols] matrix for stores: box
// [box_rows x 32] (128-byte rows), 128-byte swizzle; rows past `rows` are not written.
bool encode_f32_2d_store(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBox), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map over a row-major [rows x cols] matrix, box [box_rows x 64],
// 128-byte swizzle, out-of-bounds elements read as zero.
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

template <int S, bool BLOCK = false>
cudaError_t launch_split(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_y,
                         const PrefillParams& p, int tiles, bool pdl, cudaStream_t stream) {
    auto kernel = qkv_prefill_kernel<S, BLOCK>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Split<S>::kSmem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, (p.nt + kBM - 1) / kBM);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Split<S>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, tm_x, tm_w, tm_y, p);
}

}  // namespace

qkv_status launch_prefill(const PrefillParams& p, bool pdl, cudaStream_t stream, const char** why) {
    if (p.hd % kBN != 0) {
        *why = "head_dim must be a multiple of 64 (two 32-row boxes per neox tile)";
        return QKV_ERR_UNSUPPORTED;
    }
    if (p.H % 8 != 0) {
        *why = "hidden must be a multiple of 8 (16-byte TMA row stride)";
        return QKV_ERR_UNSUPPORTED;
    }
    if ((reinterpret_cast<uintptr_t>(p.X) | reinterpret_cast<uintptr_t>(p.W)) & 15) {
        *why = "X and W must be 16-byte aligned";
        return QKV_ERR_INVALID_ARG;
    }
    if (reinterpret_cast<uintptr_t>(p.Y) & 15) {
        *why = "Y must be 16-byte aligned";
        return QKV_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(p.kv_k) | reinterpret_cast<uintptr_t>(p.kv_v)) & 15) {
        *why = "the KV regions must be 16-byte aligned";
        return QKV_ERR_INVALID_ARG;
    }
    const int R = p.nqt + 2 * p.nkt;
    const int tiles = R / kBN;
    // Clusters of 2 pair tiles splitting K in halves when the tile count is even and K has at
    // least two 64-wide blocks, else one CTA per pair tile over the whole K range.  (Clusters
    // of 4 splitting K in quarters measured slower and are not built.)
    const int nkb = (p.H + kBK - 1) / kBK;
    const int split = tiles % 2 == 0 && nkb >= 2 ? 2 : 1;
    if (p.withhold_xchg && split != 2) {
        *why = "the exchange-timeout test needs clusters of 2 (an even count of 64-row tiles and H > 64)";
        return QKV_ERR_UNSUPPORTED;
    }
    // One 16 KB W box per K block and cluster (in place of four 4 KB boxes) when the cluster's
    // two pair tiles are 128 consecutive rows: whole heads of 64 or 128 rows, and no cluster
    // across the q|k or k|v boundary.  A bulk tensor load costs about the same time whatever
    // its size up to ~16-32 KB, so four times fewer, larger boxes stream W about 3x faster.
    const int tq = p.nqt / kBN, tk = p.nkt / kBN;
    const bool block = split == 2 && (p.hd == 64 || p.hd == 128) && tq % 2 == 0 && (tq + tk) % 2 == 0;
    CUtensorMap tm_x, tm_w, tm_y;
    if (!encode_f32_2d_store(&tm_y, p.Y, static_cast<uint64_t>(p.nt), static_cast<uint64_t>(R), kBM) ||
        !encode_bf16_2d(&tm_x, p.X, static_cast<uint64_t>(p.nt), static_cast<uint64_t>(p.H), kBM) ||
        !encode_bf16_2d(&tm_w, p.W, static_cast<uint64_t>(R), static_cast<uint64_t>(p.H),
                        block ? 2 * kBN : kBox)) {
        *why = "cuTensorMapEncodeTiled failed or is unavailable";
        return QKV_ERR_CUDA;
    }
    cudaError_t e;
    if (split == 2 && block)
        e = launch_split<2, true>(tm_x, tm_w, tm_y, p, tiles, pdl, stream);
    else if (split == 2)
        e = launch_split<2>(tm_x, tm_w, tm_y, p, tiles, pdl, stream);
    else
        e = launch_split<1>(tm_x, tm_w, tm_y, p, tiles, pdl, stream);
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return QKV_ERR_CUDA;
    }
    return QKV_OK;
}

cudaError_t prefill_status_read(cudaStream_t stream, uint32_t* flags, int32_t* bad_pos) {
    unsigned int h[2] = {0u, 0u};
    cudaError_t e = cudaMemcpyFromSymbolAsync(h, g_prefill_status, sizeof(h), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (h[0] != 0u) {
        const unsigned int zero[2] = {0u, 0u};
        e = cudaMemcpyToSymbolAsync(g_prefill_status, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return e;
    }
    *flags = h[0];
    *bad_pos = static_cast<int32_t>(h[1]);
    return cudaSuccess;
}
