/*
 * CPU oracle for the decode attention-input stage (QKV projection, bias,
 * neox RoPE, KV-cache store).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA path and never calls it; the two
 * meet only on inputs drawn from the seeded input generator.
 *
 * What it computes follows the pages:
 *   - "73 · D3-8 — G4 FusedQKV ported to CUDA", §2 (concat matmul rows
 *     wq|wk|wv, section pointers, bitwise legitimacy of the fusion) and
 *     §3.2 Excerpt A (bias add, neox pairing (j, j + hd/2), frequency
 *     freq_scale * base^(-2d/hd), angle pos * freq, rotation, KV store at
 *     pos * nkt + j, f16 conversion round-to-nearest);
 *   - "07 · The allocator: liveness, buffer reuse, and the KV cache", §2.5
 *     (per-layer K and V regions of n_ctx rows x nkt) and §3.4 (a position
 *     >= n_ctx is an error, never an overflow);
 *   - "06 · Assign + fusion — every node picks an engine, then patterns
 *     fold", §2.2 (the FFN activation: gate and up projections of the normed
 *     hidden state, SiLU(x) = x * sigmoid(x), then the elementwise product)
 *     and §2.3 (the decode FusedFFN node: one concat gate|up weight, then the
 *     SwiGLU over the two halves of its output), and §2.3 / §3 (RmsNorm, the op
 *     that produces the normed hidden state the projection reads; the pages
 *     name it without its formula, so the oracle takes the plain definition
 *     x_c = h_c * w_c / sqrt(mean(h^2) + eps)).
 *
 *   - "06 · Assign + fusion ...", §3 (the backend capability tables: FusedQkvNorm,
 *     the Qwen3 per-head-norm variant of FusedQKV, whose epilogue normalises each
 *     q and k head before the same bias / rope / store).  The pages give no
 *     formula; the oracle takes the plain reading: after the bias, each head of q
 *     (and of k) is replaced by z * w / sqrt(mean over the head's hd values of
 *     z^2 + eps), w a weight of hd values shared by the heads of q (another for
 *     k), then rotated and stored as before; v is not normalised.
 *
 * Precision: everything is carried in double; results are rounded to f32 (or
 * f32 then f16) only where the stage stores them.  Readings taken where the
 * pages are open:
 *   - the rotation angle is the f32 value RN_f32(pos * inv_freq) with
 *     inv_freq = RN_f32(freq_scale * base^(-2d/hd)) correctly rounded, and
 *     cos/sin of that f32 angle are taken in double;
 *   - the f16 cache value is RN-even of the f32 stage output (two roundings,
 *     as a round-to-nearest conversion of an f32 register does);
 *   - a position outside [0, n_ctx) stores nothing and reports status 1.
 *
 * Plain loops on purpose: no blocking, no reordering of the sums (each dot
 * product runs over c = 0 .. H-1 in order).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_POS_RANGE 1
#define ORACLE_BAD_ARG 2

/* ---- scalar conversions ------------------------------------------------ */

/* bf16 bit pattern -> value (exact: bf16 is the top half of an f32). */
double oracle_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16 encoding of f32 `f`, round to nearest, ties to even.
 * Written from the format's definition: 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; the quantum is 2^-24 below 2^-14 (subnormals) and
 * 2^(e-10) for |f| in [2^e, 2^(e+1)); magnitudes that round past 65504 become
 * infinity. */
uint16_t oracle_f32_to_f16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if ((u & 0x7F800000u) == 0x7F800000u) {                 /* inf or NaN */
        if (u & 0x007FFFFFu) return (uint16_t)(sign | 0x7E00u);
        return (uint16_t)(sign | 0x7C00u);
    }
    const double a = fabs((double)f);
    if (a == 0.0) return sign;
    int e;                                   /* a = m * 2^e with m in [0.5, 1) */
    frexp(a, &e);
    e -= 1;                                  /* a in [2^e, 2^(e+1)) */
    int qexp = (e < -14) ? -24 : e - 10;     /* log2 of the f16 quantum */
    const double q = ldexp(a, -qexp);        /* exact scaling */
    double n = floor(q);
    const double frac = q - n;
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
    /* n * 2^qexp is the rounded magnitude; encode it. */
    if (e < -14) {
        /* subnormal quantum: the code is n itself (n == 1024 is 2^-14, the
         * smallest normal, which the same formula encodes correctly). */
        return (uint16_t)(sign | (uint16_t)n);
    }
    int E = e + 15;                          /* biased exponent */
    long code = ((long)E << 10) + ((long)n - 1024); /* n in [1024, 2048] */
    if (code >= 0x7C00) return (uint16_t)(sign | 0x7C00u); /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)code);
}

/* Correctly rounded f32 frequency for pair index d of a head of width hd:
 * RN_f32(freq_scale * base^(-2d/hd)), evaluated in long double. */
float oracle_inv_freq(int d, int hd, double base, double freq_scale) {
    const long double ex = -(2.0L * (long double)d) / (long double)hd;
    const long double v = (long double)freq_scale * powl((long double)base, ex);
    return (float)v;
}

void oracle_inv_freq_table(int hd, double base, double freq_scale, float* out) {
    for (int d = 0; d < hd / 2; ++d) out[d] = oracle_inv_freq(d, hd, base, freq_scale);
}

/* Rotation angle as the f32 value RN_f32(pos * inv_freq).  The double product
 * of a 24-bit integer and a 24-bit significand is exact, so one rounding to
 * float gives the IEEE single-precision product. */
float oracle_theta(int pos, float inv_freq) {
    return (float)((double)pos * (double)inv_freq);
}

/* ---- the projection ------------------------------------------------------ */

/* y[r] = sum_{c=0}^{H-1} W[r][c] * x[c], in double, sequential in c.
 * W is row-major [R x H], f32 values (w_is_bf16 = 0) or bf16 bit patterns. */
void oracle_matvec(const void* W, int w_is_bf16, const float* x, int64_t R, int64_t H, double* y) {
    for (int64_t r = 0; r < R; ++r) {
        double acc = 0.0;
        if (w_is_bf16) {
            const uint16_t* row = (const uint16_t*)W + r * H;
            for (int64_t c = 0; c < H; ++c) acc += oracle_bf16_value(row[c]) * (double)x[c];
        } else {
            const float* row = (const float*)W + r * H;
            for (int64_t c = 0; c < H; ++c) acc += (double)row[c] * (double)x[c];
        }
        y[r] = acc;
    }
}

/* ---- the epilogue ------------------------------------------------------- */

/* One neox pair: inputs are the projected values (double) and their biases;
 * outputs are the rotated, biased values rounded to f32.
 *   x0 = y0 + b0, x1 = y1 + b1
 *   r0 = x0 cos(theta) - x1 sin(theta)
 *   r1 = x0 sin(theta) + x1 cos(theta)        */
void oracle_rope_pair(double y0, double y1, float b0, float b1, int pos, float inv_freq,
                      float* r0, float* r1) {
    const double x0 = y0 + (double)b0;
    const double x1 = y1 + (double)b1;
    const double th = (double)oracle_theta(pos, inv_freq);
    const double c = cos(th), s = sin(th);
    *r0 = (float)(x0 * c - x1 * s);
    *r1 = (float)(x0 * s + x1 * c);
}

static void kv_put(void* kv, int kv_is_f16, size_t idx, float v) {
    if (kv_is_f16) ((uint16_t*)kv)[idx] = oracle_f32_to_f16(v);
    else ((float*)kv)[idx] = v;
}

/* One token of the stage, given the projection y = [q | k | v] (double,
 * nqt + 2*nkt entries) and the concatenated bias [bq | bk | bv].
 * Writes q_out[nqt], k_out[nkt], v_out[nkt] (f32) and, when 0 <= pos < n_ctx,
 * row `pos` of the K and V regions (f32 or f16).  Returns ORACLE_POS_RANGE and
 * stores nothing in the cache for an out-of-range position. */
int oracle_qkv_token(const double* y, const float* bias, int nh, int nkv, int hd,
                     double base, double freq_scale, int pos, int n_ctx, int kv_is_f16,
                     float* q_out, float* k_out, float* v_out, void* kv_k, void* kv_v) {
    if (hd <= 0 || (hd % 2) != 0 || nh <= 0 || nkv <= 0 || n_ctx <= 0) return ORACLE_BAD_ARG;
    const int half = hd / 2;
    const int nqt = nh * hd, nkt = nkv * hd;
    const double* yq = y;
    const double* yk = y + nqt;
    const double* yv = y + nqt + nkt;
    const float* bq = bias;
    const float* bk = bias + nqt;
    const float* bv = bias + nqt + nkt;
    const int store = (pos >= 0 && pos < n_ctx);
    const size_t row = store ? (size_t)pos * (size_t)nkt : 0;

    for (int h = 0; h < nh; ++h)
        for (int d = 0; d < half; ++d) {
            const int j = h * hd + d, j2 = j + half;
            const float f = oracle_inv_freq(d, hd, base, freq_scale);
            oracle_rope_pair(yq[j], yq[j2], bq[j], bq[j2], pos, f, &q_out[j], &q_out[j2]);
        }
    for (int h = 0; h < nkv; ++h)
        for (int d = 0; d < half; ++d) {
            const int j = h * hd + d, j2 = j + half;
            const float f = oracle_inv_freq(d, hd, base, freq_scale);
            oracle_rope_pair(yk[j], yk[j2], bk[j], bk[j2], pos, f, &k_out[j], &k_out[j2]);
            if (store) {
                kv_put(kv_k, kv_is_f16, row + (size_t)j, k_out[j]);
                kv_put(kv_k, kv_is_f16, row + (size_t)j2, k_out[j2]);
            }
        }
    for (int j = 0; j < nkt; ++j) {
        v_out[j] = (float)(yv[j] + (double)bv[j]);
        if (store) kv_put(kv_v, kv_is_f16, row + (size_t)j, v_out[j]);
    }
    return store ? ORACLE_OK : ORACLE_POS_RANGE;
}

/* ---- whole-stage conveniences ------------------------------------------ */

/* Concat class: one [R x H] matrix, rows wq | wk | wv.  `y_scratch` holds R
 * doubles.  q/k/v outputs as in oracle_qkv_token. */
int oracle_qkv_decode(const void* W, int w_is_bf16, const float* x, const float* bias,
                      int hidden, int nh, int nkv, int hd, double base, double freq_scale,
                      int pos, int n_ctx, int kv_is_f16, double* y_scratch,
                      float* q_out, float* k_out, float* v_out, void* kv_k, void* kv_v) {
    const int64_t R = (int64_t)(nh + 2 * nkv) * hd;
    oracle_matvec(W, w_is_bf16, x, R, hidden, y_scratch);
    return oracle_qkv_token(y_scratch, bias, nh, nkv, hd, base, freq_scale, pos, n_ctx,
                            kv_is_f16, q_out, k_out, v_out, kv_k, kv_v);
}

/* Mixed class: three matrices wq [nqt x H], wk [nkt x H], wv [nkt x H]. */
int oracle_qkv_decode_mixed(const void* Wq, const void* Wk, const void* Wv, int w_is_bf16,
                            const float* x, const float* bias, int hidden, int nh, int nkv,
                            int hd, double base, double freq_scale, int pos, int n_ctx,
                            int kv_is_f16, double* y_scratch, float* q_out, float* k_out,
                            float* v_out, void* kv_k, void* kv_v) {
    const int64_t nqt = (int64_t)nh * hd, nkt = (int64_t)nkv * hd;
    oracle_matvec(Wq, w_is_bf16, x, nqt, hidden, y_scratch);
    oracle_matvec(Wk, w_is_bf16, x, nkt, hidden, y_scratch + nqt);
    oracle_matvec(Wv, w_is_bf16, x, nkt, hidden, y_scratch + nqt + nkt);
    return oracle_qkv_token(y_scratch, bias, nh, nkv, hd, base, freq_scale, pos, n_ctx,
                            kv_is_f16, q_out, k_out, v_out, kv_k, kv_v);
}

/* Prefill: tokens t = 0 .. nt-1 with activations X[t] (bf16 bit patterns,
 * widened exactly) at positions[t]; the per-token math is the decode stage.
 * Y is [nt x R] = per token q | k | v after the epilogue.  `x_scratch` holds
 * `hidden` floats, `y_scratch` R doubles.  Returns the first non-OK status. */
int oracle_qkv_prefill(const uint16_t* X, int nt, const void* W, int w_is_bf16,
                       const float* bias, const int32_t* positions, int hidden, int nh,
                       int nkv, int hd, double base, double freq_scale, int n_ctx,
                       int kv_is_f16, float* x_scratch, double* y_scratch, float* Y,
                       void* kv_k, void* kv_v) {
    const int64_t nqt = (int64_t)nh * hd, nkt = (int64_t)nkv * hd, R = nqt + 2 * nkt;
    int status = ORACLE_OK;
    for (int t = 0; t < nt; ++t) {
        for (int c = 0; c < hidden; ++c)
            x_scratch[c] = (float)oracle_bf16_value(X[(int64_t)t * hidden + c]);
        float* yt = Y + (int64_t)t * R;
        int s = oracle_qkv_decode(W, w_is_bf16, x_scratch, bias, hidden, nh, nkv, hd, base,
                                  freq_scale, positions[t], n_ctx, kv_is_f16, y_scratch, yt,
                                  yt + nqt, yt + nqt + nkt, kv_k, kv_v);
        if (s != ORACLE_OK && status == ORACLE_OK) status = s;
    }
    return status;
}

/* ---- FusedFFN (decode, one token) ----------------------------------------- */

/* SiLU(v) = v * sigmoid(v) = v / (1 + e^-v), in double. */
double oracle_silu(double v) { return v / (1.0 + exp(-v)); }

/* The concat gate|up projection followed by SwiGLU.
 *   W      row-major [2 nf x H]: rows 0 .. nf-1 are W_gate, rows nf .. 2nf-1 W_up
 *          (f32 values, or bf16 bit patterns when w_is_bf16).
 *   x      the normed hidden state [H].
 *   out[i] = RN_f32( silu(gate_i) * up_i ),  gate_i = (W x)[i],  up_i = (W x)[nf + i],
 *          every sum and product in double. */
void oracle_ffn_swiglu(const void* W, int w_is_bf16, const float* x, int64_t nf, int64_t H, float* out) {
    for (int64_t i = 0; i < nf; ++i) {
        double g = 0.0, u = 0.0;
        if (w_is_bf16) {
            const uint16_t* rg = (const uint16_t*)W + i * H;
            const uint16_t* ru = (const uint16_t*)W + (nf + i) * H;
            for (int64_t c = 0; c < H; ++c) {
                g += oracle_bf16_value(rg[c]) * (double)x[c];
                u += oracle_bf16_value(ru[c]) * (double)x[c];
            }
        } else {
            const float* rg = (const float*)W + i * H;
            const float* ru = (const float*)W + (nf + i) * H;
            for (int64_t c = 0; c < H; ++c) {
                g += (double)rg[c] * (double)x[c];
                u += (double)ru[c] * (double)x[c];
            }
        }
        out[i] = (float)(oracle_silu(g) * u);
    }
}

/* ---- RMSNorm of the hidden state (the step before the projection) --------- */

/* x_c = RN_f32( h_c * w_c / sqrt( (1/H) sum_j h_j^2 + eps ) ), sums and products in
 * double; x is rounded to f32 because the stage stages x in f32 before the projection. */
void oracle_rmsnorm(const float* h, const float* w, int64_t H, double eps, float* x) {
    double ss = 0.0;
    for (int64_t c = 0; c < H; ++c) ss += (double)h[c] * (double)h[c];
    const double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t c = 0; c < H; ++c) x[c] = (float)((double)h[c] * inv * (double)w[c]);
}

/* ---- FusedQkvNorm: per-head RMSNorm of q and k before the rotation -------- */

/* One head of width hd: z_i = y_i + b_i, inv = 1 / sqrt( (1/hd) sum_i z_i^2 + eps ),
 * n_i = z_i * inv * w_i, then the neox pairs (n_d, n_{d+hd/2}) rotated at `pos`.
 * Writes the rotated head (f32) to out[0 .. hd-1]. */
static void qknorm_head(const double* y, const float* b, const float* w, double eps, int hd, double base,
                        double freq_scale, int pos, float* out) {
    const int half = hd / 2;
    double ss = 0.0;
    for (int i = 0; i < hd; ++i) {
        const double z = y[i] + (double)b[i];
        ss += z * z;
    }
    const double inv = 1.0 / sqrt(ss / (double)hd + eps);
    for (int d = 0; d < half; ++d) {
        const double n0 = (y[d] + (double)b[d]) * inv * (double)w[d];
        const double n1 = (y[d + half] + (double)b[d + half]) * inv * (double)w[d + half];
        const float f = oracle_inv_freq(d, hd, base, freq_scale);
        oracle_rope_pair(n0, n1, 0.0f, 0.0f, pos, f, &out[d], &out[d + half]);
    }
}

/* One token of the FusedQkvNorm stage on the projection y = [q | k | v] (double)
 * with the concatenated bias, q_norm_w[hd] and k_norm_w[hd]: every q head and every
 * k head through qknorm_head, v biased; k and v stored at row `pos` as in
 * oracle_qkv_token (same status and range rule). */
int oracle_qkv_token_qknorm(const double* y, const float* bias, const float* q_norm_w, const float* k_norm_w,
                            double eps, int nh, int nkv, int hd, double base, double freq_scale, int pos,
                            int n_ctx, int kv_is_f16, float* q_out, float* k_out, float* v_out, void* kv_k,
                            void* kv_v) {
    if (hd <= 0 || (hd % 2) != 0 || nh <= 0 || nkv <= 0 || n_ctx <= 0 || !(eps >= 0.0)) return ORACLE_BAD_ARG;
    const int nqt = nh * hd, nkt = nkv * hd;
    const int store = (pos >= 0 && pos < n_ctx);
    const size_t row = store ? (size_t)pos * (size_t)nkt : 0;
    for (int h = 0; h < nh; ++h)
        qknorm_head(y + h * hd, bias + h * hd, q_norm_w, eps, hd, base, freq_scale, pos, q_out + h * hd);
    for (int h = 0; h < nkv; ++h) {
        qknorm_head(y + nqt + h * hd, bias + nqt + h * hd, k_norm_w, eps, hd, base, freq_scale, pos,
                    k_out + h * hd);
        if (store)
            for (int i = 0; i < hd; ++i) kv_put(kv_k, kv_is_f16, row + (size_t)(h * hd + i), k_out[h * hd + i]);
    }
    for (int j = 0; j < nkt; ++j) {
        v_out[j] = (float)(y[nqt + nkt + j] + (double)bias[nqt + nkt + j]);
        if (store) kv_put(kv_v, kv_is_f16, row + (size_t)j, v_out[j]);
    }
    return store ? ORACLE_OK : ORACLE_POS_RANGE;
}

/* Concat class: one [R x H] matrix, then oracle_qkv_token_qknorm. */
int oracle_qkv_decode_qknorm(const void* W, int w_is_bf16, const float* x, const float* bias,
                             const float* q_norm_w, const float* k_norm_w, double eps, int hidden, int nh, int nkv,
                             int hd, double base, double freq_scale, int pos, int n_ctx, int kv_is_f16,
                             double* y_scratch, float* q_out, float* k_out, float* v_out, void* kv_k, void* kv_v) {
    const int64_t R = (int64_t)(nh + 2 * nkv) * hd;
    oracle_matvec(W, w_is_bf16, x, R, hidden, y_scratch);
    return oracle_qkv_token_qknorm(y_scratch, bias, q_norm_w, k_norm_w, eps, nh, nkv, hd, base, freq_scale, pos,
                                   n_ctx, kv_is_f16, q_out, k_out, v_out, kv_k, kv_v);
}
