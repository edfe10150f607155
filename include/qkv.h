/*
 * qkv.h — C ABI of libqkv.so: the attention-input stage of transformer decode
 * on GB300 (sm_103a).
 *
 * One layer of the stage takes the normed hidden vector x and produces
 *   q = Wq x + bq,  k = Wk x + bk,  v = Wv x + bv,
 * rotates q and k with neox-paired RoPE at position pos, and stores k and v
 * into row `pos` of the layer's KV-cache regions.  Source of the definition:
 *   "73 · D3-8 — G4 FusedQKV ported to CUDA", §2 (concat weight rows wq|wk|wv,
 *   pointer-form sections, the 7-step chain bias x3 + rope x2 + store x2 and
 *   its one-launch fusion) and §3.2 Excerpt A (bias add, neox pairs
 *   (j, j + hd/2), frequency freq_scale * base^(-2d/hd), angle pos * freq,
 *   rotation, store at pos * nkt + j, f16 round-to-nearest);
 *   "07 · The allocator: liveness, buffer reuse, and the KV cache", §2.5
 *   (per-layer persistent K and V regions, n_ctx rows of nkt values).
 *
 * Conventions for every entry point:
 *   - Pointers named d_* or documented as "device" are CUDA device pointers
 *     owned by the caller.  The library never allocates, frees or retains
 *     caller memory; plans and graphs hold only host state plus, for a graph,
 *     the instantiated CUDA graph.  Pointers baked into a graph must stay
 *     valid and unmoved while the graph is used.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Work is enqueued asynchronously; the call returns before it runs.
 *   - Errors are returned, never hidden: every precondition the host can see
 *     (null pointer, bad size, wrong class, misaligned buffer, unsupported
 *     RoPE style) returns a non-zero qkv_status before anything is launched,
 *     and qkv_last_error() describes it.  There is no CPU fallback.
 *   - The position is read on the device (capture/replay safe).  A position
 *     outside [0, n_ctx) makes the kernels skip every cache store, compute the
 *     q/k/v outputs anyway, and set a device status word that
 *     qkv_check_device_error() reports; the GPU is never trapped.
 *
 * Notation: H = hidden, nh = heads, nkv = kv heads, hd = head_dim,
 * nqt = nh*hd, nkt = nkv*hd, R = nqt + 2*nkt.
 */
#ifndef QKV_H_
#define QKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QKV_ABI_VERSION 1
#define QKV_MAX_HEAD_DIM 256

typedef enum qkv_status {
    QKV_OK = 0,
    QKV_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, misaligned buffer */
    QKV_ERR_UNSUPPORTED = 2,  /* valid but not implemented: interleaved RoPE, odd hd, dtype */
    QKV_ERR_POS_RANGE = 3,    /* a host-visible position outside [0, n_ctx) */
    QKV_ERR_CUDA = 4,         /* a CUDA runtime call failed; qkv_last_error() names it */
    QKV_ERR_DEVICE_FLAG = 5   /* the device status word is set (see qkv_check_device_error) */
} qkv_status;

/* Element types.  Values are fixed and used in qkv_plan_desc's int32 fields. */
enum { QKV_F32 = 0, QKV_BF16 = 1, QKV_F16 = 2 };
/* Layer classes ("73 · D3-8 ...", §1 and §3.1): one concat matrix, or three. */
enum { QKV_CLASS_CONCAT = 0, QKV_CLASS_MIXED = 1 };
/* RoPE styles.  Only the neox (non-interleaved) pairing is implemented; the
 * page's guard rejects anything else loudly (§3.3, "The rope style guard must
 * be loud"). */
enum { QKV_ROPE_NEOX = 0, QKV_ROPE_INTERLEAVED = 1 };

/* Layer geometry and numeric formats.  All fields are 32-bit. */
typedef struct qkv_plan_desc {
    int32_t hidden;      /* H >= 1 */
    int32_t n_head;      /* nh >= 1 */
    int32_t n_head_kv;   /* nkv >= 1 */
    int32_t head_dim;    /* hd: even, 2 .. QKV_MAX_HEAD_DIM */
    float theta;         /* RoPE frequency base (> 0), 1e6 for Qwen2.5 */
    float freq_scale;    /* RoPE frequency scale (> 0), 1.0 for Qwen2.5 */
    int32_t n_ctx;       /* rows of each KV region (>= 1) */
    int32_t w_dtype;     /* QKV_F32 or QKV_BF16 weights */
    int32_t kv_dtype;    /* QKV_F32 or QKV_F16 cache */
    int32_t layer_class; /* QKV_CLASS_CONCAT or QKV_CLASS_MIXED */
    int32_t rope;        /* QKV_ROPE_NEOX (anything else: QKV_ERR_UNSUPPORTED) */
} qkv_plan_desc;

/* Sizes derived from a plan (host arithmetic only). */
typedef struct qkv_plan_info {
    int64_t rows;            /* R */
    int64_t nqt, nkt;
    int64_t pair_units;      /* R / 2: rows are produced two at a time */
    int64_t epilogue_units;  /* nqt/2 + nkt/2 + nkt: the one-launch epilogue's grid */
    int64_t weight_bytes;    /* R * H * sizeof(weight) */
    int64_t kv_row_bytes;    /* nkt * sizeof(cache element) */
    int64_t kv_region_bytes; /* n_ctx * kv_row_bytes, per region (K or V) */
    int64_t algo_bytes_decode; /* bytes one decode step must move: W + x + bias + q|k|v + 2 cache rows */
    int32_t launches_decode; /* kernel launches per decode layer: 1 for both classes */
    int32_t weight_vectorized; /* 1 if rows are streamed as 16-byte vectors */
} qkv_plan_info;

typedef struct qkv_plan qkv_plan;

/* A view of one layer's cache regions ("07 · The allocator ...", §2.5):
 * element (p, j) is at base + p * row_stride_elems + j. */
typedef struct qkv_kv_view {
    void* k;
    void* v;
    int32_t dtype;           /* QKV_F32 or QKV_F16 */
    int32_t n_ctx;
    int64_t nkt;
    int64_t row_stride_elems; /* = nkt */
    int64_t region_bytes;
} qkv_kv_view;

/* ---- library -------------------------------------------------------------- */

int qkv_abi_version(void);
const char* qkv_status_str(qkv_status s);
/* Message of the last failing call on this thread ("" if none). */
const char* qkv_last_error(void);

/* ---- plans ---------------------------------------------------------------- */

/* Validate `desc` and build a host-side plan (no CUDA call, no device memory).
 * The plan holds the RoPE frequency table inv_freq[d] = RN_f32(freq_scale *
 * theta^(-2d/hd)), correctly rounded, which every kernel receives by value.
 * Errors: INVALID_ARG (null, sizes <= 0, bad enum), UNSUPPORTED (odd hd or
 * hd > QKV_MAX_HEAD_DIM, interleaved RoPE, weight or cache dtype outside
 * {F32, BF16} / {F32, F16}).  Ownership: destroy with qkv_plan_destroy. */
qkv_status qkv_plan_create(const qkv_plan_desc* desc, qkv_plan** out);
void qkv_plan_destroy(qkv_plan* plan);
qkv_status qkv_plan_info_get(const qkv_plan* plan, qkv_plan_info* out);
/* Copy the plan's frequency table (hd/2 floats) to host memory. */
qkv_status qkv_plan_inv_freq(const qkv_plan* plan, float* out_host, int32_t n);

/* ---- decode (nt == 1) ------------------------------------------------------- */

/* Concat class, one launch: y = W x over the R rows of W = [wq; wk; wv]
 * (row-major R x H, w_dtype), then bias, RoPE on q and k, cache stores —
 * all in the projection kernel's tail ("73 · D3-8 ...", §2 and §3.2 Excerpt A).
 *   x     device, H floats.
 *   w     device, R*H weights; rows 16-byte aligned for the vector path.
 *   bias  device, R floats = bq | bk | bv.
 *   d_pos device, one int32: the position (read on the device).
 *   q,k,v device outputs: nqt, nkt, nkt floats (may be sections of one R-float
 *         buffer: q = base, k = base + nqt, v = base + nqt + nkt).  They hold
 *         the rotated q, rotated k and biased v.
 *   kv_k, kv_v device cache regions, n_ctx * nkt elements of kv_dtype; only
 *         row pos is written.
 * Errors: INVALID_ARG (null pointer, plan of the mixed class), CUDA. */
qkv_status qkv_decode_step(const qkv_plan* plan, const float* x, const void* w,
                           const float* bias, const int32_t* d_pos, float* q, float* k,
                           float* v, void* kv_k, void* kv_v, void* stream);

/* As qkv_decode_step, with the layer's RMSNorm in front (the step that produces
 * the normed hidden state the projection reads; the pages name the RmsNorm op
 * — "06 · Assign + fusion — every node picks an engine, then patterns fold",
 * §2.3 and §3 — without its formula, so this takes the plain definition):
 *   x_c = (h_c * inv) * norm_w[c],  inv = 1 / sqrt(sum_j h_j^2 / H + norm_eps),
 * computed in f32 inside the projection kernel (every CTA reduces sum(h^2) in a
 * fixed order), then y = W x as in qkv_decode_step.
 *   h       device, H floats: the hidden state before the norm.
 *   norm_w  device, H floats, 16-byte aligned.
 *   norm_eps >= 0 (Qwen2.5: 1e-6).
 * The kernel applies the scalar 1/rms to the dot products (it commutes with the
 * projection) and stages h * norm_w, so the sum of squares runs beside the
 * staging; the rounding order differs from normalising first by f32 ulps.
 * Errors: INVALID_ARG (null or misaligned norm_w, negative or NaN eps, mixed-class plan),
 * CUDA. */
qkv_status qkv_decode_step_rmsnorm(const qkv_plan* plan, const float* h, const float* norm_w,
                                   float norm_eps, const void* w, const float* bias,
                                   const int32_t* d_pos, float* q, float* k, float* v, void* kv_k,
                                   void* kv_v, void* stream);

/* Mixed class, one launch: the three projections wq (nqt x H), wk (nkt x H),
 * wv (nkt x H) and the same epilogue ("73 · D3-8 ...", §1 second complication,
 * §3.1: three matmuls without bias + one epilogue, section pointers passed in).
 * Three bias pointers (nqt, nkt, nkt floats).  Errors as qkv_decode_step. */
qkv_status qkv_decode_step_mixed(const qkv_plan* plan, const float* x, const void* wq,
                                 const void* wk, const void* wv, const float* bias_q,
                                 const float* bias_k, const float* bias_v,
                                 const int32_t* d_pos, float* q, float* k, float* v,
                                 void* kv_k, void* kv_v, void* stream);

/* Projection only (no bias, no RoPE, no store): q = wq x, k = wk x, v = wv x in
 * one launch.  For a concat plan pass wk = wq + nqt*H and wv = wk + nkt*H.  With
 * qkv_epilogue this is the page's two-launch class 1 / four-launch class 2
 * shape, kept as the comparator of the fused kernel. */
qkv_status qkv_project(const qkv_plan* plan, const float* x, const void* wq, const void* wk,
                       const void* wv, float* q, float* k, float* v, void* stream);

/* The epilogue alone, one launch over the flat index nqt/2 + nkt/2 + nkt
 * ("73 · D3-8 ...", §3.2 Excerpts A and B): q and k are biased and rotated in
 * place, v is biased in place, k and v are stored at row pos.  Pointer-form
 * sections: q/k/v and the three biases may point into concat buffers or into
 * separate ones. */
qkv_status qkv_epilogue(const qkv_plan* plan, float* q, float* k, float* v,
                        const float* bias_q, const float* bias_k, const float* bias_v,
                        const int32_t* d_pos, void* kv_k, void* kv_v, void* stream);

/* The unfused chain, one launch per call: the seven-kernel tail the page's
 * fusion replaces (bias x3, rope x2, store x2; "73 · D3-8 ...", §2).  Kept as
 * comparators: fused results must equal the chain's bit for bit.
 *   qkv_chain_add_bias: y[i] += b[i], i < n.
 *   qkv_chain_rope:     neox rotation in place of n_heads heads of hd values.
 *   qkv_chain_store:    cache[pos * nkt + j] = src[j], j < nkt (f32 or f16 RN). */
qkv_status qkv_chain_add_bias(float* y, const float* b, int64_t n, void* stream);
qkv_status qkv_chain_rope(const qkv_plan* plan, float* y, int32_t n_heads,
                          const int32_t* d_pos, void* stream);
qkv_status qkv_chain_store(const qkv_plan* plan, const float* src, void* cache,
                           const int32_t* d_pos, void* stream);

/* ---- prefill (nt >= 1) ------------------------------------------------------ */

/* Concat class, nt tokens: Y = X W^T (bf16 x bf16, f32 accumulate on the
 * tensor cores), then per token t the decode epilogue at position
 * d_positions[t].  The page keeps prefill on the unfused chain (§3.3 guards:
 * the fused epilogue is nt == 1 only); here the per-token math is the same
 * and runs in the GEMM's epilogue.  Requires w_dtype BF16.
 *   X           device, nt x H bf16 (row-major).
 *   d_positions device, nt int32, distinct positions.
 *   Y           device, nt x R floats: per token q | k | v after the epilogue.
 * X, w, Y, kv_k and kv_v must be 16-byte aligned (TMA operands and 16-byte
 * cache stores).  nt == 0 returns QKV_OK without a launch.  A token whose
 * position lies outside [0, n_ctx) still gets its Y row; its cache rows are not
 * written and bit 0 of the device status flags is set (qkv_check_device_error).
 * Errors: INVALID_ARG (null or misaligned pointers, nt < 0), UNSUPPORTED (f32
 * weights, mixed class, head_dim % 64 != 0, hidden % 8 != 0), CUDA. */
qkv_status qkv_prefill_step(const qkv_plan* plan, const uint16_t* X, int32_t nt,
                            const void* w, const float* bias, const int32_t* d_positions,
                            float* Y, void* kv_k, void* kv_v, void* stream);

/* ---- cache view ------------------------------------------------------------- */

/* Describe a layer's regions: element (p, j) at base + p * nkt + j.  Host
 * arithmetic only; the pointers are returned unchanged. */
qkv_status kv_cache_view(const qkv_plan* plan, void* kv_k, void* kv_v, qkv_kv_view* out);

/* ---- whole-model decode step in one CUDA graph ------------------------------ */

/* Per-layer buffers of a model-graph layer.  Concat layers use w and bias
 * (R rows / floats); mixed layers use wq/wk/wv and bias_q/bias_k/bias_v.
 * Outputs q/k/v and the cache regions as in qkv_decode_step. */
typedef struct qkv_layer_ptrs {
    const float* x;
    const void* w;
    const void* wq;
    const void* wk;
    const void* wv;
    const float* bias;
    const float* bias_q;
    const float* bias_k;
    const float* bias_v;
    float* q;
    float* k;
    float* v;
    void* kv_k;
    void* kv_v;
} qkv_layer_ptrs;

typedef struct qkv_graph qkv_graph;

/* Capture n_layers decode steps (plans[i] with layers[i], all reading the one
 * device position d_pos) into a CUDA graph and instantiate it.  `stream` must
 * not be the legacy default stream; it is used only for the capture.
 * Consecutive layers are chained with programmatic dependent launch: a layer
 * may start streaming its weights while the previous one finishes, and reads
 * x and writes outputs only after it completed.  Pointers are baked in.
 * Errors: INVALID_ARG, CUDA (capture or instantiation failed). */
qkv_status qkv_model_graph_create(const qkv_plan* const* plans, int32_t n_layers,
                                  const qkv_layer_ptrs* layers, const int32_t* d_pos,
                                  void* stream, qkv_graph** out);
/* As qkv_model_graph_create, with each layer's RMSNorm fused in front of its
 * projection (see qkv_decode_step_rmsnorm): layers[i].x is the hidden state
 * before the norm and norm_w[i] (device, H floats, 16-byte aligned) the layer's
 * norm weight.
 * Errors as qkv_model_graph_create, and INVALID_ARG for a null norm weight or
 * a negative / NaN eps. */
qkv_status qkv_model_graph_create_rmsnorm(const qkv_plan* const* plans, int32_t n_layers,
                                          const qkv_layer_ptrs* layers, const float* const* norm_w,
                                          float norm_eps, const int32_t* d_pos, void* stream,
                                          qkv_graph** out);
/* One decode step of the whole model: one cudaGraphLaunch on `stream`. */
qkv_status qkv_model_graph_launch(qkv_graph* graph, void* stream);
/* Copy-in, replay, copy-out on `stream`, for callers holding host buffers:
 * in_bytes from h_in (host, ideally pinned) to d_in, one replay, then
 * out_bytes from d_out to h_out.  Returns after enqueueing (synchronise
 * `stream` before reading h_out; keep h_in unchanged until then).  Either
 * byte count may be 0.  The input copy runs on a stream the graph owns
 * (created on the first call): it waits for the previous replay of this
 * graph, so it overlaps the previous call's output copy, and the replay waits
 * for it; the replay and the output copy run on `stream`. */
qkv_status qkv_model_graph_run_host(qkv_graph* graph, const void* h_in, void* d_in,
                                    size_t in_bytes, const void* d_out, void* h_out,
                                    size_t out_bytes, void* stream);
/* Per-layer buffers of a prefill graph layer (concat class, bf16 weights):
 * X [nt x H] bf16, w [R x H] bf16, bias [R], positions [nt] int32 (device),
 * Y [nt x R] f32, and the layer's cache regions — as in qkv_prefill_step. */
typedef struct qkv_prefill_ptrs {
    const uint16_t* X;
    const void* w;
    const float* bias;
    const int32_t* positions;
    float* Y;
    void* kv_k;
    void* kv_v;
} qkv_prefill_ptrs;

/* Capture n_layers prefill steps of nt tokens (plans[i] with layers[i]) into a
 * CUDA graph, chained with programmatic dependent launch; replay it with
 * qkv_model_graph_launch.  Errors as qkv_model_graph_create and
 * qkv_prefill_step. */
qkv_status qkv_prefill_graph_create(const qkv_plan* const* plans, int32_t n_layers,
                                    const qkv_prefill_ptrs* layers, int32_t nt, void* stream,
                                    qkv_graph** out);

/* ---- FusedQkvNorm decode: per-head q / k RMSNorm before the rotation -------- */

/* The Qwen3 variant of the fused stage named on page "06 · Assign + fusion —
 * every node picks an engine, then patterns fold", §3 (the backend capability
 * tables: FusedQkvNorm, "q/k per-head norm + the same bias/rope/store").  The
 * pages give no formula; this library takes the plain reading: after the
 * bias, each head of q (and of k) is replaced by
 *   z * w / sqrt( (1/hd) sum_i z_i^2 + eps ),   z = the head's hd biased values,
 * w = q_norm_w (k_norm_w for k heads, hd floats each, shared by the heads),
 * then rotated and stored exactly as in qkv_decode_step; v is not normalised.
 * f32 arithmetic throughout (sum of squares in a fixed order).
 *
 * A head's rows are computed by several CTAs, so the stage counts, per head,
 * the rows already published: the CTA that completes a head normalises,
 * rotates and stores it.  The counters live in d_workspace, caller-owned
 * device memory of qkv_qknorm_workspace_bytes() bytes (4-byte aligned) that
 * must be zero before the first call and is left zero by every completed
 * call; calls that share a workspace must not overlap on the GPU (one stream).
 * After a call that set a device status flag, zero it again. */
qkv_status qkv_qknorm_workspace_bytes(const qkv_plan* plan, size_t* out);
/* One layer, concat class (w = [wq; wk; wv], bias [R]), arguments otherwise as
 * qkv_decode_step; eps >= 0.  Rows must be 16-byte aligned (H * element size a
 * multiple of 16, x and w 16-byte aligned): else UNSUPPORTED.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
qkv_status qkv_decode_step_qknorm(const qkv_plan* plan, const float* x, const void* w, const float* bias,
                                  const float* q_norm_w, const float* k_norm_w, float eps,
                                  const int32_t* d_pos, float* q, float* k, float* v, void* kv_k,
                                  void* kv_v, void* d_workspace, void* stream);
/* qkv_decode_step_qknorm for callers that cannot allocate device memory
 * themselves (for instance code running inside an allocator callback or a
 * memory pool that must not grow, or a host that has handed every byte of the
 * GPU to another owner): the per-head counters live in a fixed array inside
 * the library (1024 counters, 4 KB, reserved on every device that loads the
 * library until the process exits), so nothing is allocated, by the caller or
 * by the library.  The pages have no counterpart of this entry point.
 *   - At most 1024 q + kv heads (nh + nkv); larger plans get INVALID_ARG.
 *   - The first call on a device looks up the array's device address there
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     device's current context; make that first call before any stream
 *     capture on the device.  After cudaDeviceReset the next call runs in a
 *     new context and looks the address up again (the same rule applies to it).
 *   - Every call clears the counters it uses (an asynchronous memset on
 *     `stream`) and shares the one array with every other call on the device:
 *     calls that may overlap on the GPU (different streams, or graph replays
 *     running concurrently) race on it.  Run them in one stream.
 * Arguments, results and other errors as qkv_decode_step_qknorm. */
qkv_status qkv_decode_step_qknorm_noalloc(const qkv_plan* plan, const float* x, const void* w, const float* bias,
                                          const float* q_norm_w, const float* k_norm_w, float eps,
                                          const int32_t* d_pos, float* q, float* k, float* v, void* kv_k,
                                          void* kv_v, void* stream);
/* The whole model in one CUDA graph as qkv_model_graph_create (either layer
 * class, programmatic dependent launch between layers), every layer through
 * the FusedQkvNorm stage with its q_norm_w[i] / k_norm_w[i]; the layers share
 * d_workspace (sized for the layer with the most heads). */
qkv_status qkv_model_graph_create_qknorm(const qkv_plan* const* plans, int32_t n_layers,
                                         const qkv_layer_ptrs* layers, const float* const* q_norm_w,
                                         const float* const* k_norm_w, float eps, const int32_t* d_pos,
                                         void* d_workspace, void* stream, qkv_graph** out);

/* ---- FusedFFN decode: the FFN's gate|up projection and SwiGLU --------------- */

/* One token of the FFN activation of page "06 · Assign + fusion — every node
 * picks an engine, then patterns fold", §2.2 (gate = W_gate x, up = W_up x of
 * the normed hidden state; SiLU(v) = v * sigmoid(v); their elementwise
 * product) in the decode form of §2.3 (one concat gate|up weight, then the
 * offset SwiGLU over the two halves of its output), as one launch:
 *   out[i] = silu(g_i) * u_i,  g_i = sum_c W[i][c] x[c],  u_i = sum_c W[nf + i][c] x[c].
 * The down projection that follows is not part of it.
 *   hidden      H (1 .. 49152).
 *   n_ff        nf, the intermediate size (>= 1).
 *   w_dtype     QKV_F32 or QKV_BF16.
 *   x           device, H floats, 16-byte aligned.
 *   w_gate_up   device, [2 nf x H] row-major: rows 0 .. nf-1 are W_gate,
 *               rows nf .. 2nf-1 W_up; 16-byte aligned.
 *   out         device, nf floats.
 * f32 accumulation over bf16 weights widened exactly; g and u are rounded to
 * f32, then silu(g) = g / (1 + e^-g) and the product are f32 operations.
 * Caller-owned memory only; nothing is allocated.
 * Errors: INVALID_ARG (null or misaligned pointers, sizes out of range),
 * UNSUPPORTED (H * element size not a multiple of 16 bytes), CUDA. */
qkv_status qkv_ffn_step(int32_t hidden, int32_t n_ff, int32_t w_dtype, const float* x,
                        const void* w_gate_up, float* out, void* stream);

/* Per-layer buffers of an FFN graph layer, as in qkv_ffn_step. */
typedef struct qkv_ffn_layer {
    const float* x;
    const void* w_gate_up;
    float* out;
} qkv_ffn_layer;

/* Capture n_layers FusedFFN steps of one shape into a CUDA graph, chained with
 * programmatic dependent launch as in qkv_model_graph_create (a layer streams
 * its weights while the previous one finishes, and reads x and writes out only
 * after it completed); replay it with qkv_model_graph_launch.  Errors as
 * qkv_model_graph_create and qkv_ffn_step. */
qkv_status qkv_ffn_graph_create(int32_t hidden, int32_t n_ff, int32_t w_dtype, int32_t n_layers,
                                const qkv_ffn_layer* layers, void* stream, qkv_graph** out);

/* Number of kernel nodes in the graph (launches per decode step). */
qkv_status qkv_model_graph_kernel_count(const qkv_graph* graph, int32_t* out);
void qkv_model_graph_destroy(qkv_graph* graph);

/* ---- device status ---------------------------------------------------------- */

/* Read (and clear) the device status word on `stream` (synchronises it).
 * flags bit 0: a kernel saw a position outside [0, n_ctx) and skipped its
 * cache stores; *bad_pos_out receives one such position.  Returns
 * QKV_ERR_DEVICE_FLAG when any flag was set, QKV_OK otherwise.  The word is
 * per device and shared by all plans. */
qkv_status qkv_check_device_error(void* stream, uint32_t* flags_out, int32_t* bad_pos_out);

#ifdef __cplusplus
}
#endif

#endif /* QKV_H_ */
