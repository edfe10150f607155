// C-ABI layer of libqkv.so: argument validation, plans, dispatch to the
// kernels, whole-model CUDA graph, device status.  See include/qkv.h for the
// contract of every entry point.
//
// Guards follow "73 · D3-8 — G4 FusedQKV ported to CUDA", §3.2 Excerpt D and
// §3.3: a failed precondition is a returned error, never a silent fallback
// (also "06 · Assign + fusion", §2.1: no mid-run fallback, ever).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "qkv_internal.h"
#include "qkv_test.h"

namespace {

thread_local std::string g_last_error;

qkv_status fail(qkv_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

qkv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(QKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int32_t dtype) { return dtype == QKV_F32 ? 4 : 2; }

// RoPE frequency of pair index d: RN_f32(freq_scale * theta^(-2d/hd)),
// evaluated in long double and rounded once ("73 · D3-8 ...", §3.2 Excerpt A
// gives the expression freq_scale / base^(2d/hd); the table fixes its f32
// value so that every kernel uses the same, correctly rounded, frequency).
float rope_inv_freq(int d, int hd, float theta, float freq_scale) {
    const long double e = -2.0L * static_cast<long double>(d) / static_cast<long double>(hd);
    return static_cast<float>(static_cast<long double>(freq_scale) *
                              powl(static_cast<long double>(theta), e));
}

DecodeParams base_params(const qkv_plan* p) {
    DecodeParams q;
    std::memset(&q, 0, sizeof q);
    q.H = p->d.hidden;
    q.nqt = static_cast<int32_t>(p->nqt);
    q.nkt = static_cast<int32_t>(p->nkt);
    q.hd = p->d.head_dim;
    q.n_ctx = p->d.n_ctx;
    q.kv_f16 = p->d.kv_dtype == QKV_F16 ? 1 : 0;
    std::memcpy(q.inv_freq, p->inv_freq, sizeof q.inv_freq);
    return q;
}

#define REQUIRE(cond, ...)                                              \
    do {                                                                \
        if (!(cond)) return fail(QKV_ERR_INVALID_ARG, __VA_ARGS__);     \
    } while (0)

qkv_status check_decode_ptrs(const qkv_plan* plan, const float* x, const void* const w[3],
                             const float* const b[3], const int32_t* d_pos, const float* q,
                             const float* k, const float* v, const void* kv_k, const void* kv_v) {
    REQUIRE(plan, "plan is null");
    REQUIRE(x, "x is null");
    REQUIRE(w[0] && w[1] && w[2], "a weight pointer is null");
    REQUIRE(b[0] && b[1] && b[2], "a bias pointer is null");
    REQUIRE(d_pos, "d_pos is null");
    REQUIRE(q && k && v, "a q/k/v output pointer is null");
    REQUIRE(kv_k && kv_v, "a KV region pointer is null");
    return QKV_OK;
}

// The vector path needs 16-byte aligned x and weight rows.
int use_vec(const qkv_plan* plan, const float* x, const void* const w[3]) {
    return plan->vec && aligned16(x) && aligned16(w[0]) && aligned16(w[1]) && aligned16(w[2]);
}

// `norm_w` non-null: x is the hidden state h and the kernel projects RMSNorm(h).
qkv_status run_decode(const qkv_plan* plan, const float* x, const void* const w[3],
                      const float* const b[3], const int32_t* d_pos, float* q, float* k, float* v,
                      void* kv_k, void* kv_v, bool pdl, cudaStream_t s, const float* norm_w = nullptr,
                      float norm_eps = 0.f, const void* const* next_w = nullptr) {
    DecodeParams p = base_params(plan);
    if (next_w != nullptr)
        for (int i = 0; i < 3; ++i) p.next_w[i] = next_w[i];
    p.norm_w = norm_w;
    p.norm_eps = norm_eps;
    p.x = x;
    for (int i = 0; i < 3; ++i) {
        p.w[i] = w[i];
        p.bias[i] = b[i];
    }
    p.out[0] = q;
    p.out[1] = k;
    p.out[2] = v;
    p.kv_k = kv_k;
    p.kv_v = kv_v;
    p.pos = d_pos;
    cudaError_t e = launch_decode(p, plan->d.w_dtype, use_vec(plan, x, w), kFused, pdl, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    return QKV_OK;
}

// FusedQkvNorm: the fused stage with per-head q / k RMSNorm; rows must be 16-byte aligned.
qkv_status check_qknorm_args(const qkv_plan* plan, const float* x, const void* const w[3], const float* q_norm_w,
                             const float* k_norm_w, float eps, const void* d_workspace) {
    REQUIRE(q_norm_w && k_norm_w, "q_norm_w or k_norm_w is null");
    REQUIRE(eps >= 0.f && eps == eps, "eps must be a number >= 0");
    REQUIRE(d_workspace, "d_workspace is null");
    REQUIRE((reinterpret_cast<uintptr_t>(d_workspace) & 3u) == 0, "d_workspace must be 4-byte aligned");
    if (!use_vec(plan, x, w))
        return fail(QKV_ERR_UNSUPPORTED, "FusedQkvNorm needs 16-byte aligned x and weight rows "
                                         "(hidden * element size a multiple of 16)");
    return QKV_OK;
}

qkv_status run_qknorm(const qkv_plan* plan, const float* x, const void* const w[3], const float* const b[3],
                      const float* q_norm_w, const float* k_norm_w, float eps, const int32_t* d_pos, float* q,
                      float* k, float* v, void* kv_k, void* kv_v, void* d_workspace, bool pdl, cudaStream_t s) {
    DecodeParams p = base_params(plan);
    p.x = x;
    for (int i = 0; i < 3; ++i) {
        p.w[i] = w[i];
        p.bias[i] = b[i];
    }
    p.out[0] = q;
    p.out[1] = k;
    p.out[2] = v;
    p.kv_k = kv_k;
    p.kv_v = kv_v;
    p.pos = d_pos;
    p.qk_norm_w[0] = q_norm_w;
    p.qk_norm_w[1] = k_norm_w;
    p.qk_eps = eps;
    p.head_cnt = static_cast<unsigned int*>(d_workspace);
    const cudaError_t e = launch_qknorm(p, plan->d.w_dtype, pdl, s);
    if (e == cudaErrorNotSupported)
        return fail(QKV_ERR_UNSUPPORTED, "hidden %d leaves no room for the ring", plan->d.hidden);
    if (e != cudaSuccess) return cuda_fail(e, "FusedQkvNorm kernel launch");
    return QKV_OK;
}

}  // namespace

// ------------------------------------------------------------------ library

extern "C" int qkv_abi_version(void) { return QKV_ABI_VERSION; }

extern "C" const char* qkv_status_str(qkv_status s) {
    switch (s) {
        case QKV_OK: return "QKV_OK";
        case QKV_ERR_INVALID_ARG: return "QKV_ERR_INVALID_ARG";
        case QKV_ERR_UNSUPPORTED: return "QKV_ERR_UNSUPPORTED";
        case QKV_ERR_POS_RANGE: return "QKV_ERR_POS_RANGE";
        case QKV_ERR_CUDA: return "QKV_ERR_CUDA";
        case QKV_ERR_DEVICE_FLAG: return "QKV_ERR_DEVICE_FLAG";
    }
    return "QKV_ERR_UNKNOWN";
}

extern "C" const char* qkv_last_error(void) { return g_last_error.c_str(); }

// ------------------------------------------------------------------ plans

extern "C" qkv_status qkv_plan_create(const qkv_plan_desc* d, qkv_plan** out) {
    REQUIRE(out, "out is null");
    *out = nullptr;
    REQUIRE(d, "desc is null");
    REQUIRE(d->hidden >= 1, "hidden must be >= 1 (got %d)", d->hidden);
    REQUIRE(d->n_head >= 1 && d->n_head_kv >= 1, "head counts must be >= 1 (got %d, %d)", d->n_head,
            d->n_head_kv);
    REQUIRE(d->head_dim >= 1, "head_dim must be >= 1 (got %d)", d->head_dim);
    REQUIRE(d->n_ctx >= 1, "n_ctx must be >= 1 (got %d)", d->n_ctx);
    REQUIRE(std::isfinite(d->theta) && d->theta > 0.f, "theta must be finite and > 0");
    REQUIRE(std::isfinite(d->freq_scale) && d->freq_scale > 0.f, "freq_scale must be finite and > 0");
    REQUIRE(d->layer_class == QKV_CLASS_CONCAT || d->layer_class == QKV_CLASS_MIXED,
            "layer_class must be QKV_CLASS_CONCAT or QKV_CLASS_MIXED (got %d)", d->layer_class);
    if (d->rope == QKV_ROPE_INTERLEAVED)
        return fail(QKV_ERR_UNSUPPORTED, "rope style INTERLEAVED is not supported: only the neox "
                                         "(non-interleaved) pairing is implemented");
    REQUIRE(d->rope == QKV_ROPE_NEOX, "unknown rope style %d", d->rope);
    if (d->head_dim % 2 != 0)
        return fail(QKV_ERR_UNSUPPORTED, "head_dim must be even for the neox pairing (got %d)", d->head_dim);
    if (d->head_dim > QKV_MAX_HEAD_DIM)
        return fail(QKV_ERR_UNSUPPORTED, "head_dim %d exceeds %d", d->head_dim, QKV_MAX_HEAD_DIM);
    if (d->w_dtype != QKV_F32 && d->w_dtype != QKV_BF16)
        return fail(QKV_ERR_UNSUPPORTED, "weight dtype %d not supported (F32 or BF16)", d->w_dtype);
    if (d->kv_dtype != QKV_F32 && d->kv_dtype != QKV_F16)
        return fail(QKV_ERR_UNSUPPORTED, "cache dtype %d not supported (F32 or F16)", d->kv_dtype);
    if (d->hidden > 49152)
        return fail(QKV_ERR_UNSUPPORTED, "hidden %d exceeds 49152 (x is staged in shared memory)", d->hidden);
    const int64_t nqt = static_cast<int64_t>(d->n_head) * d->head_dim;
    const int64_t nkt = static_cast<int64_t>(d->n_head_kv) * d->head_dim;
    const int64_t rows = nqt + 2 * nkt;
    if (rows >= (int64_t(1) << 30))
        return fail(QKV_ERR_UNSUPPORTED, "%lld projection rows exceed 2^30", static_cast<long long>(rows));
    qkv_plan* p = new (std::nothrow) qkv_plan;
    if (!p) return fail(QKV_ERR_INVALID_ARG, "out of host memory");
    std::memset(p, 0, sizeof *p);
    p->d = *d;
    p->nqt = nqt;
    p->nkt = nkt;
    p->rows = rows;
    p->half = d->head_dim / 2;
    p->vec = (static_cast<int64_t>(d->hidden) * elem_size(d->w_dtype)) % 16 == 0;
    for (int i = 0; i < d->head_dim / 2; ++i)
        p->inv_freq[i] = rope_inv_freq(i, d->head_dim, d->theta, d->freq_scale);
    *out = p;
    return QKV_OK;
}

extern "C" void qkv_plan_destroy(qkv_plan* plan) { delete plan; }

extern "C" qkv_status qkv_plan_info_get(const qkv_plan* p, qkv_plan_info* out) {
    REQUIRE(p && out, "null argument");
    const int64_t H = p->d.hidden;
    const int64_t ew = elem_size(p->d.w_dtype), ek = p->d.kv_dtype == QKV_F16 ? 2 : 4;
    out->rows = p->rows;
    out->nqt = p->nqt;
    out->nkt = p->nkt;
    out->pair_units = p->rows / 2;
    out->epilogue_units = p->nqt / 2 + p->nkt / 2 + p->nkt;
    out->weight_bytes = p->rows * H * ew;
    out->kv_row_bytes = p->nkt * ek;
    out->kv_region_bytes = out->kv_row_bytes * p->d.n_ctx;
    // W read + x read + bias read + q|k|v written + one row written in each region.
    out->algo_bytes_decode = out->weight_bytes + 4 * H + 4 * p->rows + 4 * p->rows + 2 * out->kv_row_bytes;
    out->launches_decode = 1;
    out->weight_vectorized = p->vec;
    return QKV_OK;
}

extern "C" qkv_status qkv_plan_inv_freq(const qkv_plan* p, float* out_host, int32_t n) {
    REQUIRE(p && out_host, "null argument");
    REQUIRE(n == p->d.head_dim / 2, "n must be head_dim/2 = %d", p->d.head_dim / 2);
    std::memcpy(out_host, p->inv_freq, sizeof(float) * n);
    return QKV_OK;
}

// ------------------------------------------------------------------ decode

extern "C" qkv_status qkv_decode_step(const qkv_plan* plan, const float* x, const void* w,
                                      const float* bias, const int32_t* d_pos, float* q, float* k,
                                      float* v, void* kv_k, void* kv_v, void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(plan->d.layer_class == QKV_CLASS_CONCAT,
            "qkv_decode_step needs a concat-class plan; use qkv_decode_step_mixed");
    REQUIRE(w && bias, "w or bias is null");
    const size_t es = elem_size(plan->d.w_dtype);
    const char* wb = static_cast<const char*>(w);
    const void* ws[3] = {wb, wb + plan->nqt * plan->d.hidden * es,
                         wb + (plan->nqt + plan->nkt) * plan->d.hidden * es};
    const float* bs[3] = {bias, bias + plan->nqt, bias + plan->nqt + plan->nkt};
    qkv_status st = check_decode_ptrs(plan, x, ws, bs, d_pos, q, k, v, kv_k, kv_v);
    if (st != QKV_OK) return st;
    return run_decode(plan, x, ws, bs, d_pos, q, k, v, kv_k, kv_v, false,
                      static_cast<cudaStream_t>(stream));
}

extern "C" qkv_status qkv_decode_step_rmsnorm(const qkv_plan* plan, const float* h, const float* norm_w,
                                              float norm_eps, const void* w, const float* bias,
                                              const int32_t* d_pos, float* q, float* k, float* v, void* kv_k,
                                              void* kv_v, void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(plan->d.layer_class == QKV_CLASS_CONCAT, "qkv_decode_step_rmsnorm needs a concat-class plan");
    REQUIRE(norm_w, "norm_w is null");
    REQUIRE(aligned16(norm_w), "norm_w must be 16-byte aligned");
    REQUIRE(norm_eps >= 0.f && norm_eps == norm_eps, "norm_eps must be a number >= 0");
    REQUIRE(w && bias, "w or bias is null");
    const size_t es = elem_size(plan->d.w_dtype);
    const char* wb = static_cast<const char*>(w);
    const void* ws[3] = {wb, wb + plan->nqt * plan->d.hidden * es,
                         wb + (plan->nqt + plan->nkt) * plan->d.hidden * es};
    const float* bs[3] = {bias, bias + plan->nqt, bias + plan->nqt + plan->nkt};
    qkv_status st = check_decode_ptrs(plan, h, ws, bs, d_pos, q, k, v, kv_k, kv_v);
    if (st != QKV_OK) return st;
    return run_decode(plan, h, ws, bs, d_pos, q, k, v, kv_k, kv_v, false, static_cast<cudaStream_t>(stream),
                      norm_w, norm_eps);
}

extern "C" qkv_status qkv_qknorm_workspace_bytes(const qkv_plan* plan, size_t* out) {
    REQUIRE(plan && out, "null argument");
    *out = static_cast<size_t>(plan->d.n_head + plan->d.n_head_kv) * sizeof(uint32_t);
    return QKV_OK;
}

extern "C" qkv_status qkv_decode_step_qknorm(const qkv_plan* plan, const float* x, const void* w, const float* bias,
                                             const float* q_norm_w, const float* k_norm_w, float eps,
                                             const int32_t* d_pos, float* q, float* k, float* v, void* kv_k,
                                             void* kv_v, void* d_workspace, void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(plan->d.layer_class == QKV_CLASS_CONCAT, "qkv_decode_step_qknorm needs a concat-class plan");
    REQUIRE(w && bias, "w or bias is null");
    const size_t es = elem_size(plan->d.w_dtype);
    const char* wb = static_cast<const char*>(w);
    const void* ws[3] = {wb, wb + plan->nqt * plan->d.hidden * es,
                         wb + (plan->nqt + plan->nkt) * plan->d.hidden * es};
    const float* bs[3] = {bias, bias + plan->nqt, bias + plan->nqt + plan->nkt};
    qkv_status st = check_decode_ptrs(plan, x, ws, bs, d_pos, q, k, v, kv_k, kv_v);
    if (st != QKV_OK) return st;
    st = check_qknorm_args(plan, x, ws, q_norm_w, k_norm_w, eps, d_workspace);
    if (st != QKV_OK) return st;
    return run_qknorm(plan, x, ws, bs, q_norm_w, k_norm_w, eps, d_pos, q, k, v, kv_k, kv_v, d_workspace, false,
                      static_cast<cudaStream_t>(stream));
}

extern "C" qkv_status qkv_decode_step_qknorm_noalloc(const qkv_plan* plan, const float* x, const void* w,
                                                     const float* bias, const float* q_norm_w,
                                                     const float* k_norm_w, float eps, const int32_t* d_pos,
                                                     float* q, float* k, float* v, void* kv_k, void* kv_v,
                                                     void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(plan->d.n_head + plan->d.n_head_kv <= kQknormStaticHeads,
            "qkv_decode_step_qknorm_noalloc handles at most %d q + kv heads (this plan has %d); use "
            "qkv_decode_step_qknorm with a workspace", kQknormStaticHeads, plan->d.n_head + plan->d.n_head_kv);
    REQUIRE(plan->d.layer_class == QKV_CLASS_CONCAT, "qkv_decode_step_qknorm_noalloc needs a concat-class plan");
    REQUIRE(w && bias, "w or bias is null");
    const size_t es = elem_size(plan->d.w_dtype);
    const char* wb = static_cast<const char*>(w);
    const void* ws[3] = {wb, wb + plan->nqt * plan->d.hidden * es,
                         wb + (plan->nqt + plan->nkt) * plan->d.hidden * es};
    const float* bs[3] = {bias, bias + plan->nqt, bias + plan->nqt + plan->nkt};
    qkv_status st = check_decode_ptrs(plan, x, ws, bs, d_pos, q, k, v, kv_k, kv_v);
    if (st != QKV_OK) return st;
    unsigned int* counters = nullptr;
    cudaError_t e = qknorm_static_workspace(&counters);
    if (e != cudaSuccess) return cuda_fail(e, "looking up the library's FusedQkvNorm counters");
    st = check_qknorm_args(plan, x, ws, q_norm_w, k_norm_w, eps, counters);
    if (st != QKV_OK) return st;
    // The counters must start at zero; a completed call leaves them at zero, an
    // interrupted one may not, so every call clears its share on its own stream.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(counters, 0, static_cast<size_t>(plan->d.n_head + plan->d.n_head_kv) * sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the library's FusedQkvNorm counters");
    return run_qknorm(plan, x, ws, bs, q_norm_w, k_norm_w, eps, d_pos, q, k, v, kv_k, kv_v, counters, false, s);
}

// ------------------------------------------------------------------ test hook (include/qkv_test.h)

extern "C" qkv_status qkv_test_decode_wait_timeout(const qkv_plan* plan, const float* x, const void* w,
                                                   const float* bias, const int32_t* d_pos, float* q, float* k,
                                                   float* v, void* kv_k, void* kv_v, uint32_t wait_limit_us,
                                                   void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(plan->d.layer_class == QKV_CLASS_CONCAT, "qkv_test_decode_wait_timeout needs a concat-class plan");
    REQUIRE(wait_limit_us >= 1 && wait_limit_us <= 1000, "wait_limit_us must be in [1, 1000]");
    REQUIRE(w && bias, "w or bias is null");
    const size_t es = elem_size(plan->d.w_dtype);
    const char* wb = static_cast<const char*>(w);
    const void* ws[3] = {wb, wb + plan->nqt * plan->d.hidden * es,
                         wb + (plan->nqt + plan->nkt) * plan->d.hidden * es};
    const float* bs[3] = {bias, bias + plan->nqt, bias + plan->nqt + plan->nkt};
    qkv_status st = check_decode_ptrs(plan, x, ws, bs, d_pos, q, k, v, kv_k, kv_v);
    if (st != QKV_OK) return st;
    // only the bulk-copy rings wait on copies: 16-byte aligned rows of at most 16 KB
    if (!use_vec(plan, x, ws) || static_cast<size_t>(plan->d.hidden) * es > 16384)
        return fail(QKV_ERR_UNSUPPORTED, "the wait-timeout test needs 16-byte aligned rows of at most 16 KB");
    DecodeParams p = base_params(plan);
    p.x = x;
    for (int i = 0; i < 3; ++i) {
        p.w[i] = ws[i];
        p.bias[i] = bs[i];
    }
    p.out[0] = q;
    p.out[1] = k;
    p.out[2] = v;
    p.kv_k = kv_k;
    p.kv_v = kv_v;
    p.pos = d_pos;
    p.wait_limit_ns = 1000ull * wait_limit_us;
    p.withhold_last_copy = 1;
    cudaError_t e = launch_decode(p, plan->d.w_dtype, 1, kFused, false, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    return QKV_OK;
}

extern "C" qkv_status qkv_decode_step_mixed(const qkv_plan* plan, const float* x, const void* wq,
                                            const void* wk, const void* wv, const float* bias_q,
                                            const float* bias_k, const float* bias_v,
                                            const int32_t* d_pos, float* q, float* k, float* v,
                                            void* kv_k, void* kv_v, void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(plan->d.layer_class == QKV_CLASS_MIXED,
            "qkv_decode_step_mixed needs a mixed-class plan; use qkv_decode_step");
    const void* ws[3] = {wq, wk, wv};
    const float* bs[3] = {bias_q, bias_k, bias_v};
    qkv_status st = check_decode_ptrs(plan, x, ws, bs, d_pos, q, k, v, kv_k, kv_v);
    if (st != QKV_OK) return st;
    return run_decode(plan, x, ws, bs, d_pos, q, k, v, kv_k, kv_v, false,
                      static_cast<cudaStream_t>(stream));
}

extern "C" qkv_status qkv_project(const qkv_plan* plan, const float* x, const void* wq,
                                  const void* wk, const void* wv, float* q, float* k, float* v,
                                  void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(x && wq && wk && wv, "x or a weight pointer is null");
    REQUIRE(q && k && v, "a q/k/v output pointer is null");
    DecodeParams p = base_params(plan);
    p.x = x;
    p.w[0] = wq;
    p.w[1] = wk;
    p.w[2] = wv;
    p.out[0] = q;
    p.out[1] = k;
    p.out[2] = v;
    const void* ws[3] = {wq, wk, wv};
    cudaError_t e = launch_decode(p, plan->d.w_dtype, use_vec(plan, x, ws), kProjectOnly, false,
                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "projection kernel launch");
    return QKV_OK;
}

extern "C" qkv_status qkv_epilogue(const qkv_plan* plan, float* q, float* k, float* v,
                                   const float* bias_q, const float* bias_k, const float* bias_v,
                                   const int32_t* d_pos, void* kv_k, void* kv_v, void* stream) {
    REQUIRE(plan, "plan is null");
    REQUIRE(q && k && v, "a q/k/v pointer is null");
    REQUIRE(bias_q && bias_k && bias_v, "a bias pointer is null");
    REQUIRE(d_pos, "d_pos is null");
    REQUIRE(kv_k && kv_v, "a KV region pointer is null");
    DecodeParams p = base_params(plan);
    p.bias[0] = bias_q;
    p.bias[1] = bias_k;
    p.bias[2] = bias_v;
    p.out[0] = q;
    p.out[1] = k;
    p.out[2] = v;
    p.kv_k = kv_k;
    p.kv_v = kv_v;
    p.pos = d_pos;
    cudaError_t e = launch_epilogue(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "epilogue kernel launch");
    return QKV_OK;
}

extern "C" qkv_status qkv_chain_add_bias(float* y, const float* b, int64_t n, void* stream) {
    REQUIRE(y && b, "null pointer");
    REQUIRE(n >= 0, "n must be >= 0");
    if (n == 0) return QKV_OK;
    cudaError_t e = launch_chain_add_bias(y, b, n, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "add_bias kernel launch");
    return QKV_OK;
}

extern "C" qkv_status qkv_chain_rope(const qkv_plan* plan, float* y, int32_t n_heads,
                                     const int32_t* d_pos, void* stream) {
    REQUIRE(plan && y && d_pos, "null pointer");
    REQUIRE(n_heads >= 1, "n_heads must be >= 1");
    DecodeParams p = base_params(plan);
    p.pos = d_pos;
    cudaError_t e = launch_chain_rope(p, y, n_heads, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rope kernel launch");
    return QKV_OK;
}

extern "C" qkv_status qkv_chain_store(const qkv_plan* plan, const float* src, void* cache,
                                      const int32_t* d_pos, void* stream) {
    REQUIRE(plan && src && cache && d_pos, "null pointer");
    DecodeParams p = base_params(plan);
    p.pos = d_pos;
    cudaError_t e = launch_chain_store(p, src, cache, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "store kernel launch");
    return QKV_OK;
}

// ------------------------------------------------------------------ prefill

namespace {

qkv_status check_prefill(const qkv_plan* plan, int32_t nt, const uint16_t* X, const void* w, const float* bias,
                         const int32_t* d_positions, const float* Y, const void* kv_k, const void* kv_v) {
    REQUIRE(plan, "plan is null");
    REQUIRE(nt >= 0, "nt must be >= 0");
    REQUIRE(X && w && bias && d_positions && Y && kv_k && kv_v, "null pointer");
    if (plan->d.w_dtype != QKV_BF16)
        return fail(QKV_ERR_UNSUPPORTED, "prefill needs bf16 weights (tensor-core bf16 x bf16)");
    if (plan->d.layer_class != QKV_CLASS_CONCAT)
        return fail(QKV_ERR_UNSUPPORTED, "prefill takes the concat weight matrix");
    return QKV_OK;
}

qkv_status run_prefill(const qkv_plan* plan, const uint16_t* X, int32_t nt, const void* w, const float* bias,
                       const int32_t* d_positions, float* Y, void* kv_k, void* kv_v, bool pdl,
                       cudaStream_t stream, uint64_t wait_limit_ns = 0, int32_t withhold_xchg = 0) {
    if (nt == 0) return QKV_OK;
    PrefillParams p;
    std::memset(&p, 0, sizeof p);
    p.X = X;
    p.W = static_cast<const uint16_t*>(w);
    p.bias = bias;
    p.positions = d_positions;
    p.Y = Y;
    p.kv_k = kv_k;
    p.kv_v = kv_v;
    p.nt = nt;
    p.H = plan->d.hidden;
    p.nqt = static_cast<int32_t>(plan->nqt);
    p.nkt = static_cast<int32_t>(plan->nkt);
    p.hd = plan->d.head_dim;
    p.n_ctx = plan->d.n_ctx;
    p.kv_f16 = plan->d.kv_dtype == QKV_F16 ? 1 : 0;
    p.wait_limit_ns = wait_limit_ns;
    p.withhold_xchg = withhold_xchg;
    std::memcpy(p.inv_freq, plan->inv_freq, sizeof p.inv_freq);
    const char* why = nullptr;
    qkv_status st = launch_prefill(p, pdl, stream, &why);
    if (st != QKV_OK) return fail(st, "prefill: %s", why ? why : "launch failed");
    return QKV_OK;
}

}  // namespace

extern "C" qkv_status qkv_prefill_step(const qkv_plan* plan, const uint16_t* X, int32_t nt,
                                       const void* w, const float* bias,
                                       const int32_t* d_positions, float* Y, void* kv_k,
                                       void* kv_v, void* stream) {
    qkv_status st = check_prefill(plan, nt, X, w, bias, d_positions, Y, kv_k, kv_v);
    if (st != QKV_OK) return st;
    return run_prefill(plan, X, nt, w, bias, d_positions, Y, kv_k, kv_v, false, static_cast<cudaStream_t>(stream));
}

// Test hook (include/qkv_test.h): the prefill's exchange wait made to run out.
extern "C" qkv_status qkv_test_prefill_xchg_timeout(const qkv_plan* plan, const uint16_t* X, int32_t nt,
                                                    const void* w, const float* bias, const int32_t* d_positions,
                                                    float* Y, void* kv_k, void* kv_v, uint32_t wait_limit_us,
                                                    void* stream) {
    REQUIRE(wait_limit_us >= 1 && wait_limit_us <= 1000, "wait_limit_us must be in [1, 1000]");
    qkv_status st = check_prefill(plan, nt, X, w, bias, d_positions, Y, kv_k, kv_v);
    if (st != QKV_OK) return st;
    REQUIRE(nt >= 1, "nt must be >= 1");
    return run_prefill(plan, X, nt, w, bias, d_positions, Y, kv_k, kv_v, false, static_cast<cudaStream_t>(stream),
                       1000ull * wait_limit_us, 1);
}

// ------------------------------------------------------------------ FusedFFN

namespace {

qkv_status check_ffn(int32_t H, int32_t nf, int32_t w_dtype, const float* x, const void* w, const float* out) {
    REQUIRE(H >= 1 && H <= 49152, "hidden %d out of range 1 .. 49152", H);
    REQUIRE(nf >= 1, "n_ff must be >= 1");
    REQUIRE(w_dtype == QKV_F32 || w_dtype == QKV_BF16, "w_dtype must be QKV_F32 or QKV_BF16");
    REQUIRE(x && w && out, "null x, w_gate_up or out");
    REQUIRE(aligned16(x) && aligned16(w), "x and w_gate_up must be 16-byte aligned");
    if ((static_cast<int64_t>(H) * elem_size(w_dtype)) % 16 != 0)
        return fail(QKV_ERR_UNSUPPORTED, "hidden * element size must be a multiple of 16 bytes");
    return QKV_OK;
}

qkv_status run_ffn(int32_t H, int32_t nf, int32_t w_dtype, const float* x, const void* w, float* out, bool pdl,
                   cudaStream_t s) {
    DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.x = x;
    p.w[0] = w;
    p.out[0] = out;
    p.H = H;
    p.nf = nf;
    const cudaError_t e = launch_ffn(p, w_dtype, pdl, s);
    if (e == cudaErrorNotSupported) return fail(QKV_ERR_UNSUPPORTED, "hidden %d leaves no room for the ring", H);
    if (e != cudaSuccess) return cuda_fail(e, "FusedFFN kernel launch");
    return QKV_OK;
}

}  // namespace

extern "C" qkv_status qkv_ffn_step(int32_t hidden, int32_t n_ff, int32_t w_dtype, const float* x,
                                   const void* w_gate_up, float* out, void* stream) {
    qkv_status st = check_ffn(hidden, n_ff, w_dtype, x, w_gate_up, out);
    if (st != QKV_OK) return st;
    return run_ffn(hidden, n_ff, w_dtype, x, w_gate_up, out, false, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ cache view

extern "C" qkv_status kv_cache_view(const qkv_plan* plan, void* kv_k, void* kv_v, qkv_kv_view* out) {
    REQUIRE(plan && out, "null argument");
    out->k = kv_k;
    out->v = kv_v;
    out->dtype = plan->d.kv_dtype;
    out->n_ctx = plan->d.n_ctx;
    out->nkt = plan->nkt;
    out->row_stride_elems = plan->nkt;
    out->region_bytes = plan->nkt * plan->d.n_ctx * (plan->d.kv_dtype == QKV_F16 ? 2 : 4);
    return QKV_OK;
}

// ------------------------------------------------------------------ model graph

struct qkv_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int32_t kernels = 0;
    // qkv_model_graph_run_host: the host-to-device copy runs on a stream of the graph's own,
    // after the previous replay (which reads the input block) and beside the previous
    // device-to-host copy, which stays on the caller's stream.
    cudaStream_t copy_in = nullptr;
    cudaEvent_t replayed = nullptr;  // the last replay enqueued by run_host
    cudaEvent_t copied_in = nullptr;
    cudaEvent_t copied_out = nullptr;  // the last output copy enqueued by run_host
    bool replayed_once = false;
    bool copied_out_once = false;
};

namespace {
qkv_status finish_capture(cudaStream_t s, qkv_status st, qkv_graph** out);
}

namespace {
qkv_status model_graph_create(const qkv_plan* const* plans, int32_t n_layers, const qkv_layer_ptrs* layers,
                              const float* const* norm_w, float norm_eps, const int32_t* d_pos, void* stream,
                              qkv_graph** out);
}

extern "C" qkv_status qkv_model_graph_create(const qkv_plan* const* plans, int32_t n_layers,
                                             const qkv_layer_ptrs* layers, const int32_t* d_pos,
                                             void* stream, qkv_graph** out) {
    return model_graph_create(plans, n_layers, layers, nullptr, 0.f, d_pos, stream, out);
}

extern "C" qkv_status qkv_model_graph_create_rmsnorm(const qkv_plan* const* plans, int32_t n_layers,
                                                     const qkv_layer_ptrs* layers, const float* const* norm_w,
                                                     float norm_eps, const int32_t* d_pos, void* stream,
                                                     qkv_graph** out) {
    REQUIRE(out, "out is null");
    *out = nullptr;
    REQUIRE(norm_w, "norm_w is null");
    REQUIRE(norm_eps >= 0.f && norm_eps == norm_eps, "norm_eps must be a number >= 0");
    for (int32_t i = 0; i < n_layers; ++i) {
        REQUIRE(norm_w[i], "norm weight of layer %d is null", i);
        REQUIRE(aligned16(norm_w[i]), "norm weight of layer %d must be 16-byte aligned", i);
    }
    return model_graph_create(plans, n_layers, layers, norm_w, norm_eps, d_pos, stream, out);
}

namespace {
// Section pointers of a model-graph layer (both classes).
void layer_sections(const qkv_plan* p, const qkv_layer_ptrs& L, const void* ws[3], const float* bs[3]) {
    if (p->d.layer_class == QKV_CLASS_CONCAT) {
        const size_t es = elem_size(p->d.w_dtype);
        const char* wb = static_cast<const char*>(L.w);
        ws[0] = wb;
        ws[1] = wb + p->nqt * p->d.hidden * es;
        ws[2] = wb + (p->nqt + p->nkt) * p->d.hidden * es;
        bs[0] = L.bias;
        bs[1] = L.bias + p->nqt;
        bs[2] = L.bias + p->nqt + p->nkt;
    } else {
        ws[0] = L.wq;
        ws[1] = L.wk;
        ws[2] = L.wv;
        bs[0] = L.bias_q;
        bs[1] = L.bias_k;
        bs[2] = L.bias_v;
    }
}
}  // namespace

extern "C" qkv_status qkv_model_graph_create_qknorm(const qkv_plan* const* plans, int32_t n_layers,
                                                    const qkv_layer_ptrs* layers, const float* const* q_norm_w,
                                                    const float* const* k_norm_w, float eps, const int32_t* d_pos,
                                                    void* d_workspace, void* stream, qkv_graph** out) {
    REQUIRE(out, "out is null");
    *out = nullptr;
    REQUIRE(plans && layers && d_pos && q_norm_w && k_norm_w, "null argument");
    REQUIRE(n_layers >= 1, "n_layers must be >= 1");
    REQUIRE(stream, "capture needs a non-default stream");
    for (int32_t i = 0; i < n_layers; ++i) {
        const qkv_plan* p = plans[i];
        const qkv_layer_ptrs& L = layers[i];
        REQUIRE(p, "plan of layer %d is null", i);
        if (p->d.layer_class == QKV_CLASS_CONCAT) {
            REQUIRE(L.w && L.bias, "layer %d (concat): w or bias is null", i);
        } else {
            REQUIRE(L.wq && L.wk && L.wv && L.bias_q && L.bias_k && L.bias_v,
                    "layer %d (mixed): a weight or bias pointer is null", i);
        }
        const void* ws[3];
        const float* bs[3];
        layer_sections(p, L, ws, bs);
        qkv_status st = check_decode_ptrs(p, L.x, ws, bs, d_pos, L.q, L.k, L.v, L.kv_k, L.kv_v);
        if (st == QKV_OK) st = check_qknorm_args(p, L.x, ws, q_norm_w[i], k_norm_w[i], eps, d_workspace);
        if (st != QKV_OK) return fail(st, "layer %d: %s", i, g_last_error.c_str());
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
    qkv_status st = QKV_OK;
    for (int32_t i = 0; i < n_layers && st == QKV_OK; ++i) {
        const qkv_layer_ptrs& L = layers[i];
        const void* ws[3];
        const float* bs[3];
        layer_sections(plans[i], L, ws, bs);
        st = run_qknorm(plans[i], L.x, ws, bs, q_norm_w[i], k_norm_w[i], eps, d_pos, L.q, L.k, L.v, L.kv_k, L.kv_v,
                        d_workspace, i > 0, s);
    }
    return finish_capture(s, st, out);
}

namespace {
qkv_status model_graph_create(const qkv_plan* const* plans, int32_t n_layers, const qkv_layer_ptrs* layers,
                              const float* const* norm_w, float norm_eps, const int32_t* d_pos, void* stream,
                              qkv_graph** out) {
    REQUIRE(out, "out is null");
    *out = nullptr;
    REQUIRE(plans && layers && d_pos, "null argument");
    REQUIRE(n_layers >= 1, "n_layers must be >= 1");
    REQUIRE(stream, "capture needs a non-default stream");
    // Validate every layer before capturing anything.
    for (int32_t i = 0; i < n_layers; ++i) {
        const qkv_plan* p = plans[i];
        const qkv_layer_ptrs& L = layers[i];
        REQUIRE(p, "plan of layer %d is null", i);
        if (p->d.layer_class == QKV_CLASS_CONCAT) {
            REQUIRE(L.w && L.bias, "layer %d (concat): w or bias is null", i);
        } else {
            REQUIRE(L.wq && L.wk && L.wv && L.bias_q && L.bias_k && L.bias_v,
                    "layer %d (mixed): a weight or bias pointer is null", i);
        }
        REQUIRE(L.x && L.q && L.k && L.v && L.kv_k && L.kv_v, "layer %d: null x/q/k/v/kv pointer", i);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
    qkv_status st = QKV_OK;
    for (int32_t i = 0; i < n_layers && st == QKV_OK; ++i) {
        const qkv_plan* p = plans[i];
        const qkv_layer_ptrs& L = layers[i];
        const void* ws[3];
        const float* bs[3];
        if (p->d.layer_class == QKV_CLASS_CONCAT) {
            const size_t es = elem_size(p->d.w_dtype);
            const char* wb = static_cast<const char*>(L.w);
            ws[0] = wb;
            ws[1] = wb + p->nqt * p->d.hidden * es;
            ws[2] = wb + (p->nqt + p->nkt) * p->d.hidden * es;
            bs[0] = L.bias;
            bs[1] = L.bias + p->nqt;
            bs[2] = L.bias + p->nqt + p->nkt;
        } else {
            ws[0] = L.wq;
            ws[1] = L.wk;
            ws[2] = L.wv;
            bs[0] = L.bias_q;
            bs[1] = L.bias_k;
            bs[2] = L.bias_v;
        }
        // the next layer's weights, when it has this layer's shape, as an L2 prefetch hint
        const void* nws[3] = {nullptr, nullptr, nullptr};
        if (i + 1 < n_layers) {
            const qkv_plan* q = plans[i + 1];
            const float* nbs[3];
            if (q->d.hidden == p->d.hidden && q->nqt == p->nqt && q->nkt == p->nkt && q->d.w_dtype == p->d.w_dtype)
                layer_sections(q, layers[i + 1], nws, nbs);
        }
        st = run_decode(p, L.x, ws, bs, d_pos, L.q, L.k, L.v, L.kv_k, L.kv_v, i > 0, s,
                        norm_w ? norm_w[i] : nullptr, norm_eps, nws[0] != nullptr ? nws : nullptr);
    }
    return finish_capture(s, st, out);
}
}  // namespace

namespace {

// End a capture started by one of the graph builders, count its kernel nodes and
// instantiate it.  `st` is the status of the launches made during the capture.
qkv_status finish_capture(cudaStream_t s, qkv_status st, qkv_graph** out) {
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (st != QKV_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
    size_t n_nodes = 0;
    e = cudaGraphGetNodes(graph, nullptr, &n_nodes);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaGraphGetNodes");
    }
    std::vector<cudaGraphNode_t> nodes(n_nodes);
    int32_t kernels = 0;
    if (n_nodes) {
        e = cudaGraphGetNodes(graph, nodes.data(), &n_nodes);
        if (e != cudaSuccess) {
            cudaGraphDestroy(graph);
            return cuda_fail(e, "cudaGraphGetNodes");
        }
        for (size_t i = 0; i < n_nodes; ++i) {
            cudaGraphNodeType t;
            if (cudaGraphNodeGetType(nodes[i], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kernels;
        }
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return cuda_fail(e, "cudaGraphInstantiate");
    }
    qkv_graph* g = new (std::nothrow) qkv_graph;
    if (!g) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return fail(QKV_ERR_INVALID_ARG, "out of host memory");
    }
    g->graph = graph;
    g->exec = exec;
    g->kernels = kernels;
    *out = g;
    return QKV_OK;
}

}  // namespace

extern "C" qkv_status qkv_ffn_graph_create(int32_t hidden, int32_t n_ff, int32_t w_dtype, int32_t n_layers,
                                           const qkv_ffn_layer* layers, void* stream, qkv_graph** out) {
    REQUIRE(out, "out is null");
    *out = nullptr;
    REQUIRE(layers, "layers is null");
    REQUIRE(n_layers >= 1, "n_layers must be >= 1");
    REQUIRE(stream, "capture needs a non-default stream");
    for (int32_t i = 0; i < n_layers; ++i) {
        qkv_status st = check_ffn(hidden, n_ff, w_dtype, layers[i].x, layers[i].w_gate_up, layers[i].out);
        if (st != QKV_OK) return fail(st, "layer %d: %s", i, g_last_error.c_str());
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
    qkv_status st = QKV_OK;
    for (int32_t i = 0; i < n_layers && st == QKV_OK; ++i)
        st = run_ffn(hidden, n_ff, w_dtype, layers[i].x, layers[i].w_gate_up, layers[i].out, i > 0, s);
    return finish_capture(s, st, out);
}

extern "C" qkv_status qkv_prefill_graph_create(const qkv_plan* const* plans, int32_t n_layers,
                                               const qkv_prefill_ptrs* layers, int32_t nt, void* stream,
                                               qkv_graph** out) {
    REQUIRE(out, "out is null");
    *out = nullptr;
    REQUIRE(plans && layers, "null argument");
    REQUIRE(n_layers >= 1, "n_layers must be >= 1");
    REQUIRE(nt >= 1, "nt must be >= 1");
    REQUIRE(stream, "capture needs a non-default stream");
    for (int32_t i = 0; i < n_layers; ++i) {
        const qkv_prefill_ptrs& L = layers[i];
        qkv_status st = check_prefill(plans[i], nt, L.X, L.w, L.bias, L.positions, L.Y, L.kv_k, L.kv_v);
        if (st != QKV_OK) return fail(st, "layer %d: %s", i, g_last_error.c_str());
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
    qkv_status st = QKV_OK;
    for (int32_t i = 0; i < n_layers && st == QKV_OK; ++i) {
        const qkv_prefill_ptrs& L = layers[i];
        st = run_prefill(plans[i], L.X, nt, L.w, L.bias, L.positions, L.Y, L.kv_k, L.kv_v, i > 0, s);
    }
    return finish_capture(s, st, out);
}

extern "C" qkv_status qkv_model_graph_launch(qkv_graph* g, void* stream) {
    REQUIRE(g, "graph is null");
    cudaError_t e = cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
    return QKV_OK;
}

extern "C" qkv_status qkv_model_graph_run_host(qkv_graph* g, const void* h_in, void* d_in,
                                               size_t in_bytes, const void* d_out, void* h_out,
                                               size_t out_bytes, void* stream) {
    REQUIRE(g, "graph is null");
    REQUIRE(in_bytes == 0 || (h_in && d_in), "null input buffer");
    REQUIRE(out_bytes == 0 || (h_out && d_out), "null output buffer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!g->copy_in) {
        e = cudaStreamCreateWithFlags(&g->copy_in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->replayed, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->copied_in, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->copied_out, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "creating the graph's copy stream");
    }
    if (in_bytes) {
        // The input block may be overwritten once the previous replay has read it; the
        // previous call's device-to-host copy (on the caller's stream) runs meanwhile.
        if (g->replayed_once) {
            e = cudaStreamWaitEvent(g->copy_in, g->replayed, 0);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
        }
        e = cudaMemcpyAsync(d_in, h_in, in_bytes, cudaMemcpyHostToDevice, g->copy_in);
        if (e == cudaSuccess) e = cudaEventRecord(g->copied_in, g->copy_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, g->copied_in, 0);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    }
    if (g->copied_out_once) {
        // the replay overwrites the outputs the previous call copies out (whatever its stream)
        e = cudaStreamWaitEvent(s, g->copied_out, 0);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
    }
    e = cudaGraphLaunch(g->exec, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
    e = cudaEventRecord(g->replayed, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    g->replayed_once = true;
    if (out_bytes) {
        e = cudaMemcpyAsync(h_out, d_out, out_bytes, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaEventRecord(g->copied_out, s);
        if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
        g->copied_out_once = true;
    }
    return QKV_OK;
}

extern "C" qkv_status qkv_model_graph_kernel_count(const qkv_graph* g, int32_t* out) {
    REQUIRE(g && out, "null argument");
    *out = g->kernels;
    return QKV_OK;
}

extern "C" void qkv_model_graph_destroy(qkv_graph* g) {
    if (!g) return;
    if (g->copy_in) {
        cudaStreamSynchronize(g->copy_in);
        cudaStreamDestroy(g->copy_in);
    }
    if (g->replayed) cudaEventDestroy(g->replayed);
    if (g->copied_in) cudaEventDestroy(g->copied_in);
    if (g->copied_out) cudaEventDestroy(g->copied_out);
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
}

// ------------------------------------------------------------------ device status

extern "C" qkv_status qkv_check_device_error(void* stream, uint32_t* flags_out, int32_t* bad_pos_out) {
    uint32_t flags = 0, pflags = 0;
    int32_t bad = 0, pbad = 0;
    cudaError_t e = device_status_read(static_cast<cudaStream_t>(stream), &flags, &bad);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    e = prefill_status_read(static_cast<cudaStream_t>(stream), &pflags, &pbad);
    if (e != cudaSuccess) return cuda_fail(e, "reading the prefill status word");
    if (!flags) bad = pbad;
    flags |= pflags;
    if (flags_out) *flags_out = flags;
    if (bad_pos_out) *bad_pos_out = bad;
    if (flags) return fail(QKV_ERR_DEVICE_FLAG, "device status flags 0x%x (position %d outside [0, n_ctx))",
                           flags, bad);
    return QKV_OK;
}
