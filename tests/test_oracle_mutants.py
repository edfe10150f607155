"""Planted mistakes in copies of the oracle must each fail at least one pin.

Every mutant is a textual edit of ``oracle/qkv_oracle.c`` compiled into a
temporary library on the CPU; the real oracle is never modified.  This shows
that the pins constrain each part of the oracle: projection, frequency,
rotation, sections, bias, cache addressing and f16 rounding.
"""
import os

import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "qkv_oracle.c")

MUTANTS = {
    "rotation_sign": ("*r0 = (float)(x0 * c - x1 * s);", "*r0 = (float)(x0 * c + x1 * s);"),
    "cos_sin_swapped": ("const double c = cos(th), s = sin(th);",
                        "const double c = sin(th), s = cos(th);"),
    "interleaved_pairs": ("const int j = h * hd + d, j2 = j + half;",
                          "const int j = h * hd + 2 * d, j2 = j + 1;"),
    "qk_bias_dropped": ("const double x0 = y0 + (double)b0;", "const double x0 = y0;"),
    "v_bias_dropped": ("v_out[j] = (float)(yv[j] + (double)bv[j]);", "v_out[j] = (float)(yv[j]);"),
    "v_offset_2nkt": ("const double* yv = y + nqt + nkt;", "const double* yv = y + 2 * nkt;"),
    "freq_exponent": ("-(2.0L * (long double)d)", "-((long double)d)"),
    "freq_not_rounded_f32": ("return (float)v;", "return (float)(double)(v * 1.0000001L);"),
    "kv_row_stride": ("(size_t)pos * (size_t)nkt : 0;", "(size_t)pos * (size_t)(nkt - 1) : 0;"),
    "kv_stores_wrong_value": ("kv_put(kv_k, kv_is_f16, row + (size_t)j2, k_out[j2]);",
                              "kv_put(kv_k, kv_is_f16, row + (size_t)j2, k_out[j]);"),
    "f16_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;",
                      "if (frac >= 0.5) n += 1.0;"),
    "f16_truncates": ("if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;",
                      "(void)frac;"),
    "matvec_drops_last_bf16": ("for (int64_t c = 0; c < H; ++c) acc += oracle_bf16_value",
                               "for (int64_t c = 0; c < H - 1; ++c) acc += oracle_bf16_value"),
    "matvec_drops_last_f32": ("for (int64_t c = 0; c < H; ++c) acc += (double)row[c]",
                              "for (int64_t c = 0; c + 1 < H; ++c) acc += (double)row[c]"),
    "matvec_transposed": ("acc += (double)row[c] * (double)x[c];",
                          "acc += (double)((const float*)W)[c * R + r] * (double)x[c];"),
    "angle_in_double": ("return (float)((double)pos * (double)inv_freq);",
                        "return (float)((double)pos * (double)inv_freq * (1.0 + 1e-7));"),
    "stage_skips_k_rope": ("oracle_rope_pair(yk[j], yk[j2], bk[j], bk[j2], pos, f,",
                           "oracle_rope_pair(yk[j], yk[j2], bk[j], bk[j2], 0, f,"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "silu_is_sigmoid": ("return v / (1.0 + exp(-v));", "return 1.0 / (1.0 + exp(-v));"),
    "ffn_gate_up_swapped": ("out[i] = (float)(oracle_silu(g) * u);", "out[i] = (float)(oracle_silu(u) * g);"),
    "ffn_up_row_reversed": ("const float* ru = (const float*)W + (nf + i) * H;",
                            "const float* ru = (const float*)W + (2 * nf - 1 - i) * H;"),
    "ffn_up_row_reversed_bf16": ("const uint16_t* ru = (const uint16_t*)W + (nf + i) * H;",
                                 "const uint16_t* ru = (const uint16_t*)W + (2 * nf - 1 - i) * H;"),
    "rmsnorm_sum_not_mean": ("const double inv = 1.0 / sqrt(ss / (double)H + eps);",
                             "const double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_eps_outside_root": ("const double inv = 1.0 / sqrt(ss / (double)H + eps);",
                                 "const double inv = 1.0 / (sqrt(ss / (double)H) + eps);"),
    "rmsnorm_weight_dropped": ("x[c] = (float)((double)h[c] * inv * (double)w[c]);",
                               "x[c] = (float)((double)h[c] * inv);"),
    "rmsnorm_no_root": ("const double inv = 1.0 / sqrt(ss / (double)H + eps);",
                        "const double inv = 1.0 / (ss / (double)H + eps);"),
    "qknorm_mean_over_2hd": ("const double inv = 1.0 / sqrt(ss / (double)hd + eps);",
                             "const double inv = 1.0 / sqrt(ss / (double)(2 * hd) + eps);"),
    "qknorm_eps_dropped": ("const double inv = 1.0 / sqrt(ss / (double)hd + eps);",
                           "const double inv = 1.0 / sqrt(ss / (double)hd);"),
    "qknorm_no_root": ("const double inv = 1.0 / sqrt(ss / (double)hd + eps);",
                       "const double inv = 1.0 / (ss / (double)hd + eps);"),
    "qknorm_bias_not_in_rms": ("const double z = y[i] + (double)b[i];", "const double z = y[i];"),
    "qknorm_weight_index": ("const double n1 = (y[d + half] + (double)b[d + half]) * inv * (double)w[d + half];",
                            "const double n1 = (y[d + half] + (double)b[d + half]) * inv * (double)w[d];"),
    "qknorm_k_uses_q_weight": ("qknorm_head(y + nqt + h * hd, bias + nqt + h * hd, k_norm_w,",
                               "qknorm_head(y + nqt + h * hd, bias + nqt + h * hd, q_norm_w,"),
    "qknorm_rotation_skipped": ("oracle_rope_pair(n0, n1, 0.0f, 0.0f, pos, f, &out[d], &out[d + half]);",
                                "oracle_rope_pair(n0, n1, 0.0f, 0.0f, 0, f, &out[d], &out[d + half]);"),
    "qknorm_k_not_stored": ("for (int i = 0; i < hd; ++i) kv_put(kv_k, kv_is_f16, row + (size_t)(h * hd + i), k_out[h * hd + i]);",
                            "for (int i = 0; i + 1 < hd; ++i) kv_put(kv_k, kv_is_f16, row + (size_t)(h * hd + i), k_out[h * hd + i]);"),
    "freq_scale_ignored": ("const long double v = (long double)freq_scale * powl((long double)base, ex);",
                           "const long double v = powl((long double)base, ex);"),
    "q_freq_index_shifted": ("const float f = oracle_inv_freq(d, hd, base, freq_scale);\n            oracle_rope_pair(yq[j]",
                             "const float f = oracle_inv_freq(d + 1, hd, base, freq_scale);\n            oracle_rope_pair(yq[j]"),
    "out_of_range_reports_ok": ("return store ? ORACLE_OK : ORACLE_POS_RANGE;", "return ORACLE_OK;"),
    "prefill_every_token_reads_x0": ("x_scratch[c] = (float)oracle_bf16_value(X[(int64_t)t * hidden + c]);",
                                     "x_scratch[c] = (float)oracle_bf16_value(X[c]);"),
    "prefill_first_position_only": ("freq_scale, positions[t], n_ctx, kv_is_f16, y_scratch, yt,",
                                    "freq_scale, positions[0], n_ctx, kv_is_f16, y_scratch, yt,"),
    "mixed_wk_wv_swapped": ("oracle_matvec(Wk, w_is_bf16, x, nkt, hidden, y_scratch + nqt);",
                            "oracle_matvec(Wv, w_is_bf16, x, nkt, hidden, y_scratch + nqt);"),
    "ffn_drops_last_column": ("for (int64_t c = 0; c < H; ++c) {\n                g += (double)rg[c]",
                              "for (int64_t c = 0; c + 1 < H; ++c) {\n                g += (double)rg[c]"),
    # wiring of the concat FusedQkvNorm wrapper (projection rows, scratch, norm weights, position)
    "qknorm_wrapper_rows_short": ("const int64_t R = (int64_t)(nh + 2 * nkv) * hd;\n    oracle_matvec(W, w_is_bf16, x, R, hidden, y_scratch);\n    return oracle_qkv_token_qknorm(",
                                  "const int64_t R = (int64_t)(nh + nkv) * hd;\n    oracle_matvec(W, w_is_bf16, x, R, hidden, y_scratch);\n    return oracle_qkv_token_qknorm("),
    "qknorm_wrapper_norm_weights_swapped": ("return oracle_qkv_token_qknorm(y_scratch, bias, q_norm_w, k_norm_w,",
                                            "return oracle_qkv_token_qknorm(y_scratch, bias, k_norm_w, q_norm_w,"),
    "qknorm_wrapper_scratch_offset": ("return oracle_qkv_token_qknorm(y_scratch, bias,",
                                      "return oracle_qkv_token_qknorm(y_scratch + hd, bias,"),
    "qknorm_wrapper_position_dropped": ("eps, nh, nkv, hd, base, freq_scale, pos,\n                                   n_ctx,",
                                        "eps, nh, nkv, hd, base, freq_scale, 0,\n                                   n_ctx,"),
    "qknorm_v_from_2nkt": ("v_out[j] = (float)(y[nqt + nkt + j] + (double)bias[nqt + nkt + j]);",
                           "v_out[j] = (float)(y[2 * nkt + j] + (double)bias[nqt + nkt + j]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: update the mutant table"
    mut_src = tmp_path / ("oracle_%s.c" % name)
    mut_src.write_text(src.replace(old, new))
    lib_path = oracle.build(force=True, src=str(mut_src), out=str(tmp_path / ("lib_%s.so" % name)))
    orc = oracle.Oracle(oracle.load(lib_path))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "planted mistake %r passed every pin" % name
