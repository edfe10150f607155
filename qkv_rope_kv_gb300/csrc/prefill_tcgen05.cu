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
// Tiling.  One CTA computes a tile of 128 tokens (UMMA M) x 64 weight rows
// (UMMA N).  The 64 rows are two 32-row boxes chosen so that every neox pair
// lands in one thread: for a q or k tile, rows (h*hd + d0 .. +31) and
// (h*hd + hd/2 + d0 .. +31); for a v tile, 64 consecutive rows.  K advances in
// blocks of 64 bf16 (128 bytes, one 128B-swizzle row).  CTAs of a thread-block
// cluster (CN consecutive row tiles, same tokens) share X: each loads a 1/CN
// slice of every X stage with TMA multicast, so one L2 read feeds CN CTAs.
// Warp 0 lane 0 streams W boxes into a 6-stage ring (before the dependency wait:
// weights are parameters) and warp 2 lane 0 its X slices into a 4-stage ring
// (mbarrier transaction counts; an X stage is reused once all CN CTAs of the
// cluster released it);
// warp 1 lane 0 issues tcgen05.mma (kind::f16, bf16 x bf16 -> f32 in TMEM,
// 4 MMAs of K = 16 per block) and releases each stage in every CTA of the cluster
// with a multicast tcgen05.commit; then
// all four warps read their 32 TMEM lanes (one token each) with tcgen05.ld and
// run the epilogue: Y leaves through shared memory (128-byte swizzle) and two
// TMA tensor stores, the token's k/v cache rows as 16-byte stores.  Every wait
// is bounded; on expiry the kernel flags the device status word, drains
// in-flight copies and MMAs, frees TMEM and returns.  A CTA leaves only after a
// cluster barrier, so no peer still writes into it.
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
#ifndef QKV_PREFILL_KSUB
#define QKV_PREFILL_KSUB 2
#endif
#ifndef QKV_PREFILL_X_STAGES
#define QKV_PREFILL_X_STAGES 4
#endif
#ifndef QKV_PREFILL_W_STAGES
#define QKV_PREFILL_W_STAGES 6
#endif
// A stage holds kSub consecutive 64-wide K blocks, so each weight row is
// requested kSub * 128 contiguous bytes at a time.  X (L2-resident, shared by
// the cluster) and W (streamed from HBM) have rings of their own: W, the long-
// latency stream, gets the deeper one.
constexpr int kSub = QKV_PREFILL_KSUB;
constexpr int kXStages = QKV_PREFILL_X_STAGES;
constexpr int kWStages = QKV_PREFILL_W_STAGES;
constexpr int kThreads = 128;
constexpr uint32_t kABlk = kBM * kBK * 2;      // 16 KB: one X block (128 x 64)
constexpr uint32_t kBBlk = kBN * kBK * 2;      // 8 KB: one W block (64 x 64)
constexpr uint32_t kABytes = kSub * kABlk;     // X bytes per stage
constexpr uint32_t kBBytes = kSub * kBBlk;     // W bytes per stage
constexpr uint32_t kBoxBytes = kBox * kBK * 2; // 4 KB
constexpr uint32_t kTmemCols = 64;             // f32 accumulator columns (= kBN)
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kXStages * kABytes + kWStages * kBBytes +
                              (2 * kXStages + 2 * kWStages + 1) * sizeof(uint64_t) + 16;
static_assert(kSmemBytes <= 227 * 1024, "prefill rings exceed shared memory");

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

// The same box into the same shared-memory offset of every CTA in `mask`; each
// destination CTA's barrier at `bar`'s offset receives the bytes it got.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                               uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(mask)
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

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
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

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, N = 64, M = 128.
constexpr uint32_t kIdesc = (1u << 4)             // D format: f32
                            | (1u << 7)           // A format: bf16
                            | (1u << 10)          // B format: bf16
                            | ((kBN >> 3) << 17)  // N >> 3
                            | ((kBM >> 4) << 24); // M >> 4

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Arrive once on the barrier at `bar`'s offset in every CTA of `mask` when the
// MMAs issued so far have completed.
__device__ __forceinline__ void tc_commit_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
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

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- kernel

__global__ void __launch_bounds__(kThreads, 1)
    qkv_prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ PrefillParams p, int cn) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ float bias_s[kBN];
    __shared__ float freq_s[kBox];
    __shared__ uint32_t tmem_slot;
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* sA = smem;                          // X ring
    unsigned char* sB = smem + kXStages * kABytes;     // W ring
    uint64_t* xfull = reinterpret_cast<uint64_t*>(sB + kWStages * kBBytes);
    uint64_t* xempty = xfull + kXStages;
    uint64_t* wfull = xempty + kXStages;
    uint64_t* wempty = wfull + kWStages;
    uint64_t* done = wempty + kWStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kBM;
    const int half = p.hd >> 1;
    const int tiles_per_head = p.hd / kBN;
    const int tq = p.nqt / kBN, tk = p.nkt / kBN;
    const int tile = blockIdx.x;
    int sec, rowA, rowB, d0;  // section and section-local first rows of the two boxes
    if (tile < tq + tk) {
        sec = tile < tq ? 0 : 1;
        const int v = sec ? tile - tq : tile;
        const int h = v / tiles_per_head;
        d0 = (v - h * tiles_per_head) * kBox;
        rowA = h * p.hd + d0;
        rowB = rowA + half;
    } else {
        sec = 2;
        d0 = 0;
        rowA = (tile - tq - tk) * kBN;
        rowB = rowA + kBox;
    }
    const int base = sec == 0 ? 0 : (sec == 1 ? p.nqt : p.nqt + p.nkt);  // section's first global row
    const int nk = (p.H + kSub * kBK - 1) / (kSub * kBK);  // stages of kSub K blocks
    // Clusters start their K loop at different blocks, so the X tiles read at any
    // moment are spread over L2; the CTAs of one cluster share X and move together.
#ifndef QKV_PREFILL_STAGGER
#define QKV_PREFILL_STAGGER 1
#endif
    const int k_first =
        QKV_PREFILL_STAGGER ? static_cast<int>((static_cast<long long>(cluster_id_x()) * nk) / cluster_count_x()) : 0;
    const uint32_t rank = cluster_rank();
    const uint16_t cmask = static_cast<uint16_t>((1u << cn) - 1u);
    const int slice = kBM / cn;  // X rows this CTA loads (and multicasts) per block

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < kXStages; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], static_cast<uint32_t>(cn));  // one release from each CTA of the cluster
        }
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], 1);
        }
        mbar_init(done, 1);
        mbar_fence_init();
    }
    if (threadIdx.x < kBox) bias_s[threadIdx.x] = p.bias[base + rowA + threadIdx.x];
    else if (threadIdx.x < 2 * kBox) bias_s[threadIdx.x] = p.bias[base + rowB + threadIdx.x - kBox];
    else if (threadIdx.x < 3 * kBox && sec < 2) freq_s[threadIdx.x - 2 * kBox] = p.inv_freq[d0 + threadIdx.x - 2 * kBox];
    tc_fence_before();
    // every barrier of the cluster is initialised before any peer copies or commits to it
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    // The next grid may be scheduled now (it waits for this one before it reads
    // anything this one writes).  X, positions and the outputs may belong to the
    // preceding grid in the stream: every thread waits for it before touching
    // them.  Weights are parameters, so the W producer streams them first.
    griddep_launch_dependents();
    if (!(warp == 0 && lane == 0)) griddep_wait();

    if (warp == 0 && lane == 0) {
        // ---- W producer: two 32 x 64 boxes per K block, local ring ----
        prefetch_tensormap(&tm_w);
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kWStages;
            if (kb >= kWStages && !mbar_wait_bounded(&wempty[s], ((kb / kWStages) - 1) & 1)) {
                flag_timeout();
                break;
            }
            const int kx = (k_first + kb) % nk;  // stage index along K
            mbar_arrive_expect_tx(&wfull[s], kBBytes);
#pragma unroll
            for (int j = 0; j < kSub; ++j) {
                const int kc = (kx * kSub + j) * kBK;  // element column of this 64-wide block
                unsigned char* b = sB + s * kBBytes + j * kBBlk;
                tma_load_2d(b, &tm_w, kc, base + rowA, &wfull[s]);
                tma_load_2d(b + kBoxBytes, &tm_w, kc, base + rowB, &wfull[s]);
            }
            ++issued;
        }
        // Drain: every W copy has landed and the MMAs released the last stages.
        const int first = issued > kWStages ? issued - kWStages : 0;
        for (int kb = first; kb < issued; ++kb) {
            if (!mbar_wait_bounded(&wfull[kb % kWStages], (kb / kWStages) & 1)) flag_timeout();
            if (!mbar_wait_bounded(&wempty[kb % kWStages], (kb / kWStages) & 1)) flag_timeout();
        }
        griddep_wait();  // before this thread writes its epilogue rows
    } else if (warp == 2 && lane == 0) {
        // ---- X producer: this CTA's slice of each 128 x 64 X block, multicast to the cluster ----
        prefetch_tensormap(&tm_x);
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kXStages;
            if (kb >= kXStages && !mbar_wait_bounded(&xempty[s], ((kb / kXStages) - 1) & 1)) {
                flag_timeout();
                break;
            }
            const int kx = (k_first + kb) % nk;
            mbar_arrive_expect_tx(&xfull[s], kABytes);  // the whole block: every CTA's slice lands here
#pragma unroll
            for (int j = 0; j < kSub; ++j) {
                unsigned char* a = sA + s * kABytes + j * kABlk + static_cast<uint32_t>(rank) * slice * (kBK * 2);
                const int kc = (kx * kSub + j) * kBK;
                if (cn == 1)
                    tma_load_2d(a, &tm_x, kc, m0, &xfull[s]);
                else
                    tma_load_2d_mc(a, &tm_x, kc, m0 + static_cast<int>(rank) * slice, &xfull[s], cmask);
            }
            ++issued;
        }
        // Drain: every slice into this CTA (its own and its peers') has landed, and
        // every CTA of the cluster released the last stages, so no peer commit is
        // still on its way to these barriers.
        const int first = issued > kXStages ? issued - kXStages : 0;
        for (int kb = first; kb < issued; ++kb) {
            if (!mbar_wait_bounded(&xfull[kb % kXStages], (kb / kXStages) & 1)) flag_timeout();
            if (!mbar_wait_bounded(&xempty[kb % kXStages], (kb / kXStages) & 1)) flag_timeout();
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        for (int kb = 0; kb < nk; ++kb) {
            const int xs = kb % kXStages, ws = kb % kWStages;
            if (!mbar_wait_bounded(&xfull[xs], (kb / kXStages) & 1) ||
                !mbar_wait_bounded(&wfull[ws], (kb / kWStages) & 1)) {
                flag_timeout();
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < kSub; ++j) {
                const unsigned char* a = sA + xs * kABytes + j * kABlk;
                const unsigned char* b = sB + ws * kBBytes + j * kBBlk;
#pragma unroll
                for (int k = 0; k < kBK / kUK; ++k)
                    tc_mma(tmem, smem_desc_k128(a + k * kUK * 2), smem_desc_k128(b + k * kUK * 2),
                           (kb | j | k) != 0);
            }
            // Both stages are free in this CTA once these MMAs have read them; an X
            // stage must be freed by every CTA of the cluster before a peer reloads it.
            tc_commit(&wempty[ws]);
            if (cn == 1)
                tc_commit(&xempty[xs]);
            else
                tc_commit_mc(&xempty[xs], cmask);
        }
        tc_commit(done);  // arrives when every MMA issued above has completed
    }
    __syncwarp();

    // ---- epilogue: thread (warp, lane) owns TMEM lane 32*warp + lane = token m0 + that ----
    // Warp-uniform: tcgen05.ld below is a warp-collective instruction.
    const bool acc_ready = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(done, 0));
    if (!acc_ready && lane == 0) flag_timeout();
    tc_fence_after();
    float acc[kBN];
    if (acc_ready) {
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        tc_ld_32cols(taddr, acc);
        tc_ld_32cols(taddr + kBox, acc + kBox);
        tc_wait_ld();
    }
    const int tl = warp * 32 + lane;  // this thread's token within the tile
    const int t = m0 + tl;
    if (acc_ready) {
        const bool live = t < p.nt;
        const int pos = live ? p.positions[t] : 0;
        const bool store = live && pos_ok(pos, p.n_ctx);
        if (live && !store) flag_bad_pos(pos);
        if (sec < 2) {
#pragma unroll
            for (int i = 0; i < kBox; ++i) {
                const float x0 = __fadd_rn(acc[i], bias_s[i]);
                const float x1 = __fadd_rn(acc[kBox + i], bias_s[kBox + i]);
                float r0, r1;
                rope_rotate(x0, x1, rope_theta(pos, freq_s[i]), r0, r1);
                acc[i] = r0;
                acc[kBox + i] = r1;
            }
        } else {
#pragma unroll
            for (int i = 0; i < kBN; ++i) acc[i] = __fadd_rn(acc[i], bias_s[i]);
        }
        // Y: stage both 32-column boxes in the (now idle) ring, row tl of each box,
        // in the 128-byte-swizzled layout the Y tensor map stores from.
        float* ys = reinterpret_cast<float*>(smem);
#pragma unroll
        for (int c = 0; c < kBox / 4; ++c) {
            const int sw = (c ^ (tl & 7)) * 4;
            *reinterpret_cast<float4*>(ys + tl * kBox + sw) =
                make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
            *reinterpret_cast<float4*>(ys + kBM * kBox + tl * kBox + sw) =
                make_float4(acc[kBox + 4 * c], acc[kBox + 4 * c + 1], acc[kBox + 4 * c + 2], acc[kBox + 4 * c + 3]);
        }
        // k and v rows of the cache: 16-byte stores of this token's two 32-column runs.
        if (store && sec > 0) {
            const size_t kvrow = static_cast<size_t>(pos) * static_cast<size_t>(p.nkt);
            void* kv = sec == 1 ? p.kv_k : p.kv_v;
            if (p.kv_f16) {
                __half* dst = static_cast<__half*>(kv) + kvrow;
#pragma unroll
                for (int c = 0; c < kBox / 8; ++c) {
                    uint4 ua, ub;
                    uint32_t* pa = &ua.x;
                    uint32_t* pb = &ub.x;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pa[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[8 * c + 2 * e]))) |
                                (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[8 * c + 2 * e + 1]))) << 16);
                        pb[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[kBox + 8 * c + 2 * e]))) |
                                (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[kBox + 8 * c + 2 * e + 1])))
                                 << 16);
                    }
                    *reinterpret_cast<uint4*>(dst + rowA + 8 * c) = ua;
                    *reinterpret_cast<uint4*>(dst + rowB + 8 * c) = ub;
                }
            } else {
                float* dst = static_cast<float*>(kv) + kvrow;
#pragma unroll
                for (int c = 0; c < kBox / 4; ++c) {
                    *reinterpret_cast<float4*>(dst + rowA + 4 * c) =
                        make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
                    *reinterpret_cast<float4*>(dst + rowB + 4 * c) = make_float4(
                        acc[kBox + 4 * c], acc[kBox + 4 * c + 1], acc[kBox + 4 * c + 2], acc[kBox + 4 * c + 3]);
                }
            }
        }
    }
    fence_proxy_async_smem();
    // Every warp has staged its rows (or the accumulator never became ready).
    const bool tile_ready = __syncthreads_and(acc_ready) != 0;
    if (tile_ready && threadIdx.x == 0) {
        const float* ys = reinterpret_cast<const float*>(smem);
        tma_store_2d(&tm_y, ys, base + rowA, m0);
        tma_store_2d(&tm_y, ys + kBM * kBox, base + rowB, m0);
        bulk_commit_and_wait_read();  // the boxes are read out before the CTA lets go of its shared memory
    }
    tc_fence_before();
    // No CTA leaves while a peer of its cluster may still write into it.
    cluster_sync_all();
    if (warp == 0) {
        // After a timeout, give in-flight MMAs a second bounded wait before the
        // accumulator columns are released.
        if (!acc_ready) mbar_wait_bounded(done, 0);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
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
    // Cluster of CN consecutive row tiles sharing X: the largest of 4, 2, 1 that divides the tiles.
#ifndef QKV_PREFILL_CLUSTER
#define QKV_PREFILL_CLUSTER 4
#endif
    int cn = QKV_PREFILL_CLUSTER;
    while (cn > 1 && tiles % cn != 0) cn >>= 1;
    CUtensorMap tm_x, tm_w, tm_y;
    if (!encode_f32_2d_store(&tm_y, p.Y, static_cast<uint64_t>(p.nt), static_cast<uint64_t>(R), kBM) ||
        !encode_bf16_2d(&tm_x, p.X, static_cast<uint64_t>(p.nt), static_cast<uint64_t>(p.H),
                        static_cast<uint32_t>(kBM / cn)) ||
        !encode_bf16_2d(&tm_w, p.W, static_cast<uint64_t>(R), static_cast<uint64_t>(p.H), kBox)) {
        *why = "cuTensorMapEncodeTiled failed or is unavailable";
        return QKV_ERR_CUDA;
    }
    cudaError_t e = cudaFuncSetAttribute(qkv_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) {
        *why = cudaGetErrorString(e);
        return QKV_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, (p.nt + kBM - 1) / kBM);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cn);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, qkv_prefill_kernel, tm_x, tm_w, tm_y, p, cn);
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
