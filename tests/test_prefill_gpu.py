"""Prefill (tcgen05 GEMM + per-token epilogue) against the CPU oracle through the C ABI.

Shapes cover a single token, tokens fewer than one M tile, several M tiles with a
ragged tail, K not a multiple of the 64-element K block (TMA zero fill), head_dim
64 and 128, f32 and f16 caches, and the Qwen2.5-14B prefill workload (nt = 128,
positions 0..127, 48 layers): full comparison on four layers, sampled tokens on
the rest.  nt = 1 prefill equals the decode oracle; out-of-range positions set
the device status flag and store nothing.
"""
import concurrent.futures as cf

import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import PREFILL_RMS_FLOOR, assert_f32_close, assert_kv_region, canary, to_dev, to_host
from qkv_rope_kv_gb300 import configs, synth

pytestmark = pytest.mark.gpu

DT = {"f32": Q.QKV_F32, "f16": Q.QKV_F16}


def run_prefill(H, nh, nkv, hd, n_ctx, kvdt, X, W, b, positions, kk0, vv0, theta=1e6):
    import torch
    plan = Q.qkv_plan_create(H, nh, nkv, hd, theta, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=DT[kvdt])
    nt = X.shape[0]
    R = (nh + 2 * nkv) * hd
    dY = torch.full((nt, R), float("nan"), dtype=torch.float32, device="cuda")
    dk, dv = to_dev(kk0), to_dev(vv0)
    dpos = torch.from_numpy(np.asarray(positions, np.int32)).cuda()
    Q.qkv_prefill_step(plan, to_dev(X), nt, to_dev(W), to_dev(b), dpos, dY, dk, dv)
    torch.cuda.synchronize()
    kvt = np.float32 if kvdt == "f32" else np.uint16
    return to_host(dY), to_host(dk, kvt), to_host(dv, kvt)


def oracle_prefill(orc, X, W, b, positions, nh, nkv, hd, kk0, vv0, theta=1e6, tokens=None, threads=16):
    """Per-token oracle (tokens in parallel threads; each writes its own cache row)."""
    kk, vv = kk0.copy(), vv0.copy()
    nt = X.shape[0]
    tokens = range(nt) if tokens is None else tokens
    out = {}

    def one(t):
        x = (X[t].astype(np.uint32) << 16).view(np.float32)
        st, q, k, v = orc.decode(W, x, b, nh, nkv, hd, theta, 1.0, int(positions[t]), kk, vv)
        return t, st, np.concatenate([q, k, v])

    with cf.ThreadPoolExecutor(threads) as ex:
        for t, st, y in ex.map(one, tokens):
            out[t] = (st, y)
    return out, kk, vv


def check(nh, nkv, hd, got, want, positions, what):
    Y, dk, dv = got
    res, kk, vv = want
    nqt, nkt = nh * hd, nkv * hd
    for t, (st, y) in res.items():
        assert st == 0
        assert_f32_close(Y[t, :nqt], y[:nqt], "%s token %d q" % (what, t), floor=PREFILL_RMS_FLOOR)
        assert_f32_close(Y[t, nqt:nqt + nkt], y[nqt:nqt + nkt], "%s token %d k" % (what, t),
                         floor=PREFILL_RMS_FLOOR)
        assert_f32_close(Y[t, nqt + nkt:], y[nqt + nkt:], "%s token %d v" % (what, t), floor=PREFILL_RMS_FLOOR)
    # rows of every token were written; compare the checked tokens' rows and require
    # every row that no token writes to keep its bits
    checked = [int(positions[t]) for t in res]
    unchecked = sorted(set(int(p) for p in positions) - set(checked))
    keep = np.ones(dk.shape[0], bool)
    keep[unchecked] = False
    rows = [int(np.sum(keep[:r])) for r in checked]
    assert_kv_region(dk[keep], kk[keep], rows, what + " K", floor=PREFILL_RMS_FLOOR)
    assert_kv_region(dv[keep], vv[keep], rows, what + " V", floor=PREFILL_RMS_FLOOR)
    # every token's cache rows (checked or not) hold exactly its k and v outputs, rounded
    # to the cache type (f16 round-to-nearest-even is numpy's float32 -> float16 cast)
    for t in range(Y.shape[0]):
        p = int(positions[t])
        if not 0 <= p < dk.shape[0]:
            continue
        ky, vy = Y[t, nqt:nqt + nkt], Y[t, nqt + nkt:]
        if dk.dtype == np.uint16:
            ky, vy = ky.astype(np.float16).view(np.uint16), vy.astype(np.float16).view(np.uint16)
        assert np.array_equal(dk[p].view(ky.dtype), ky), "%s: K row %d is not token %d's k" % (what, p, t)
        assert np.array_equal(dv[p].view(vy.dtype), vy), "%s: V row %d is not token %d's v" % (what, p, t)


SHAPES = [
    # nt, H, nh, nkv, hd, n_ctx, kv
    (1, 64, 2, 1, 64, 4, "f16"),
    (5, 128, 2, 1, 64, 16, "f32"),
    (130, 1000, 2, 2, 64, 300, "f16"),      # K tail of 40 elements, M tail of 2 tokens
    (128, 1024, 4, 2, 128, 256, "f32"),
    (37, 5120, 40, 8, 128, 4096, "f16"),    # 14B layer shape
    (3, 256, 3, 1, 64, 8, "f16"),           # 5 row tiles: no cluster sharing
    (9, 512, 1, 1, 64, 12, "f32"),          # 3 row tiles: no cluster sharing
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "nt%d_H%d_h%d_kv%d_d%d_%s" % (s[:5] + (s[6],)))
def test_prefill_matches_oracle(orc, qkv, shape):
    nt, H, nh, nkv, hd, n_ctx, kvdt = shape
    R = (nh + 2 * nkv) * hd
    W = synth.weight_rows(0, 11, 0, R, H, "bf16")
    b = synth.bias(0, 11, R)
    X = synth.prefill_x(0, 11, nt, H)
    rng = np.random.default_rng(nt + H)
    positions = rng.permutation(n_ctx)[:nt].astype(np.int32)
    kk0, vv0 = canary(n_ctx, nkv * hd, kvdt, 21), canary(n_ctx, nkv * hd, kvdt, 22)
    got = run_prefill(H, nh, nkv, hd, n_ctx, kvdt, X, W, b, positions, kk0, vv0)
    want = oracle_prefill(orc, X, W, b, positions, nh, nkv, hd, kk0, vv0)
    check(nh, nkv, hd, got, want, positions, "prefill %s" % (shape,))
    assert Q.qkv_check_device_error()[0] == 0


def test_prefill_single_token_equals_decode(orc, qkv):
    """nt = 1: the tensor-core path and the decode oracle agree at the same position."""
    import torch
    H, nh, nkv, hd, n_ctx, pos = 896, 14, 2, 64, 64, 17
    R = (nh + 2 * nkv) * hd
    W = synth.weight_rows(0, 12, 0, R, H, "bf16")
    b = synth.bias(0, 12, R)
    X = synth.prefill_x(0, 12, 1, H)
    kk0 = np.zeros((n_ctx, nkv * hd), np.uint16)
    got = run_prefill(H, nh, nkv, hd, n_ctx, "f16", X, W, b, [pos], kk0, kk0.copy())
    x = (X[0].astype(np.uint32) << 16).view(np.float32)
    kk, vv = kk0.copy(), kk0.copy()
    st, q, k, v = orc.decode(W, x, b, nh, nkv, hd, 1e6, 1.0, pos, kk, vv)
    assert_f32_close(got[0][0], np.concatenate([q, k, v]), "nt=1 prefill vs decode oracle",
                     floor=PREFILL_RMS_FLOOR)
    # and against the GPU decode kernel on the same inputs
    plan = Q.qkv_plan_create(H, nh, nkv, hd, 1e6, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16)
    out = torch.empty(R, dtype=torch.float32, device="cuda")
    dk = torch.zeros(n_ctx, nkv * hd, dtype=torch.int16, device="cuda")
    dv = torch.zeros_like(dk)
    Q.qkv_decode_step(plan, to_dev(x), to_dev(W), to_dev(b), torch.tensor([pos], dtype=torch.int32, device="cuda"),
                      out[:nh * hd], out[nh * hd:(nh + nkv) * hd], out[(nh + nkv) * hd:], dk, dv)
    torch.cuda.synchronize()
    assert_f32_close(got[0][0], to_host(out), "nt=1 prefill vs GPU decode", floor=PREFILL_RMS_FLOOR)


def test_prefill_out_of_range_position(orc, qkv):
    nt, H, nh, nkv, hd, n_ctx = 4, 256, 2, 1, 64, 8
    R = (nh + 2 * nkv) * hd
    W = synth.weight_rows(0, 13, 0, R, H, "bf16")
    b = synth.bias(0, 13, R)
    X = synth.prefill_x(0, 13, nt, H)
    positions = np.array([1, 9, 3, -2], np.int32)  # 9 and -2 outside [0, 8)
    kk0, vv0 = canary(n_ctx, nkv * hd, "f16", 31), canary(n_ctx, nkv * hd, "f16", 32)
    Q.qkv_check_device_error()
    Y, dk, dv = run_prefill(H, nh, nkv, hd, n_ctx, "f16", X, W, b, positions, kk0, vv0)
    flags, bad = Q.qkv_check_device_error()
    assert flags & 1 and bad in (9, -2)
    res, kk, vv = oracle_prefill(orc, X, W, b, positions, nh, nkv, hd, kk0, vv0)
    for t in range(nt):
        assert_f32_close(Y[t], res[t][1], "token %d" % t, floor=PREFILL_RMS_FLOOR)
    assert_kv_region(dk, kk, [1, 3], "K", floor=PREFILL_RMS_FLOOR)
    assert_kv_region(dv, vv, [1, 3], "V", floor=PREFILL_RMS_FLOOR)


@pytest.mark.slow
def test_qwen14b_prefill_nt128_48_layers(orc, qkv):
    """The 14B prefill workload: every layer on the GPU, caches filled with per-slot canaries;
    the oracle checks all 128 tokens of layers 0, 23, 24 and 47 and 8 sampled tokens of
    every other layer; on every layer the 3968 rows no token writes keep their canary bits
    and every token's cache rows hold its own k and v outputs."""
    w = configs.QWEN14B_PREFILL
    R, H = w.rows, w.hidden
    positions = np.arange(w.nt, dtype=np.int32)
    rng = np.random.default_rng(5)
    for layer in range(w.n_layers):
        W = synth.weight_rows(0, layer, 0, R, H, "bf16")
        b = synth.bias(0, layer, R)
        X = synth.prefill_x(0, layer, w.nt, H)
        kk0, vv0 = canary(w.n_ctx, w.nkt, "f16", 2 * layer), canary(w.n_ctx, w.nkt, "f16", 2 * layer + 1)
        got = run_prefill(H, w.n_head, w.n_head_kv, w.head_dim, w.n_ctx, "f16", X, W, b, positions, kk0, vv0)
        tokens = range(w.nt) if layer in (0, 23, 24, 47) else sorted(rng.choice(w.nt, 8, replace=False))
        want = oracle_prefill(orc, X, W, b, positions, w.n_head, w.n_head_kv, w.head_dim, kk0, vv0,
                              tokens=tokens)
        check(w.n_head, w.n_head_kv, w.head_dim, got, want, positions, "14B prefill layer %d" % layer)
    assert Q.qkv_check_device_error()[0] == 0


def test_prefill_graph_equals_sequential_calls(qkv):
    """Three prefill layers captured in one graph (PDL-chained) give the bits of three
    separate qkv_prefill_step calls; the graph has one kernel per layer."""
    import torch
    nt, H, nh, nkv, hd, n_ctx, L = 64, 512, 4, 2, 64, 128, 3
    R = (nh + 2 * nkv) * hd
    plan = Q.qkv_plan_create(H, nh, nkv, hd, 1e6, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16)
    positions = torch.arange(10, 10 + nt, dtype=torch.int32, device="cuda")
    layers = []
    for l in range(L):
        layers.append(dict(X=to_dev(synth.prefill_x(0, 40 + l, nt, H)), w=to_dev(synth.weight_rows(0, 40 + l, 0, R, H, "bf16")),
                           bias=to_dev(synth.bias(0, 40 + l, R)), positions=positions,
                           Y=torch.zeros(nt, R, dtype=torch.float32, device="cuda"),
                           kv_k=torch.zeros(n_ctx, nkv * hd, dtype=torch.int16, device="cuda"),
                           kv_v=torch.zeros(n_ctx, nkv * hd, dtype=torch.int16, device="cuda")))
    stream = torch.cuda.Stream()
    g = Q.qkv_prefill_graph_create([plan] * L, layers, nt, stream)
    assert g.kernel_count == L
    g.launch(stream)
    stream.synchronize()
    first = [(to_host(d["Y"]).copy(), to_host(d["kv_k"]).copy(), to_host(d["kv_v"]).copy()) for d in layers]
    for d in layers:
        d["Y"].zero_(); d["kv_k"].zero_(); d["kv_v"].zero_()
    torch.cuda.synchronize()
    for d in layers:
        Q.qkv_prefill_step(plan, d["X"], nt, d["w"], d["bias"], d["positions"], d["Y"], d["kv_k"], d["kv_v"])
    torch.cuda.synchronize()
    for d, (y, k, v) in zip(layers, first):
        assert np.array_equal(to_host(d["Y"]).view(np.uint32), y.view(np.uint32))
        assert np.array_equal(to_host(d["kv_k"]), k) and np.array_equal(to_host(d["kv_v"]), v)
