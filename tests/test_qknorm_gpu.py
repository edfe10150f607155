"""FusedQkvNorm on the GPU against the oracle: the fused stage with every q and k head
RMS-normalised (weights of hd values, after the bias, before the rotation; page "06 ·
Assign + fusion — every node picks an engine, then patterns fold", §3, plain reading of the
per-head norm).  Shapes: Qwen3-14B, -8B and -0.6B layers (rows of 10, 8 and 2 KB: both ring
configurations), f32 weights, head widths 6 (a ragged last unit per head) and 256, heads
spread over several CTAs; two calls in a row on one workspace (the per-head counters come
back to zero); an out-of-range position; the graph (both layer classes) against steps bit
for bit; and the 48-layer Qwen3-14B-shape graph, every layer against the oracle."""
import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import HostLayer, assert_f32_close, assert_kv_region, canary, to_dev, to_host
from qkv_rope_kv_gb300 import synth
from test_decode_gpu import compare, kv_np, make_plan

pytestmark = pytest.mark.gpu

EPS = 1e-6
THETA = 1e6

SHAPES = [
    # H, nh, nkv, hd, w dtype, kv dtype, n_ctx, pos
    (5120, 40, 8, 128, "bf16", "f16", 4096, 3254),  # Qwen3-14B layer (10 KB rows: large ring)
    (4096, 32, 8, 128, "bf16", "f16", 4096, 1641),  # Qwen3-8B layer (8 KB rows)
    (1024, 16, 8, 128, "bf16", "f16", 512, 100),    # Qwen3-0.6B layer (2 KB rows: small ring)
    (2048, 16, 4, 128, "f32", "f32", 64, 7),        # f32 rows of 8 KB
    (1000, 7, 3, 6, "bf16", "f16", 300, 257),       # hd 6: 3 pairs per head, ragged last unit
    (2048, 4, 2, 256, "bf16", "f16", 64, 9),        # hd 256 (the widest head)
]


def norm_weights(hd, layer):
    return synth.qk_norm_weights(0, layer, hd)


def workspace(plan):
    import torch
    n = Q.qkv_qknorm_workspace_bytes(plan) // 4
    return torch.zeros(n, dtype=torch.int32, device="cuda")


def run_qknorm(L, plan, x, qnw, knw, pos, kk0, vv0, ws, calls=1):
    import torch
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    dW, db, dx = to_dev(L.W), to_dev(L.bias), to_dev(x)
    dq, dk_w = to_dev(qnw), to_dev(knw)
    outs = []
    for _ in range(calls):
        out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
        dk, dv = to_dev(kk0), to_dev(vv0)
        q, k, v = out[:L.nqt], out[L.nqt:L.nqt + L.nkt], out[L.nqt + L.nkt:]
        Q.qkv_decode_step_qknorm(plan, dx, dW, db, dq, dk_w, EPS, dpos, q, k, v, dk, dv, ws)
        torch.cuda.synchronize()
        kvt = kv_np("f32" if plan.desc.kv_dtype == Q.QKV_F32 else "f16")
        outs.append((to_host(out), to_host(dk, kvt), to_host(dv, kvt)))
    return outs


def oracle_qknorm(orc, L, x, qnw, knw, pos, kk0, vv0):
    kk, vv = kk0.copy(), vv0.copy()
    st, q, k, v = orc.decode_qknorm(L.W, x, L.bias, qnw, knw, EPS, L.nh, L.nkv, L.hd, THETA, 1.0, pos, kk, vv)
    return st, np.concatenate([q, k, v]), kk, vv


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_h%d_kv%d_d%d_%s_%s" % s[:6])
def test_qknorm_matches_oracle(orc, qkv, shape):
    H, nh, nkv, hd, wdt, kvdt, n_ctx, pos = shape
    L = HostLayer(H, nh, nkv, hd, wdt, layer=3)
    x = L.x(pos)
    qnw, knw = norm_weights(hd, 3)
    kk0, vv0 = canary(n_ctx, L.nkt, kvdt, 21), canary(n_ctx, L.nkt, kvdt, 22)
    plan = make_plan(L, kvdt, n_ctx, wdt, theta=THETA)
    ws = workspace(plan)
    first, second = run_qknorm(L, plan, x, qnw, knw, pos, kk0, vv0, ws, calls=2)
    want = oracle_qknorm(orc, L, x, qnw, knw, pos, kk0, vv0)
    assert want[0] == 0
    compare(L, first, want, pos, "qknorm %s" % (shape,))
    # the same workspace again: identical bits, and its counters are back at zero
    for a, b in zip(first, second):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert not to_host(ws).any()
    assert Q.qkv_check_device_error()[0] == 0


def test_qknorm_position_out_of_range(orc, qkv):
    """pos = n_ctx: q/k/v are still the normalised, rotated values, no cache row is written,
    and the device status reports the position."""
    H, nh, nkv, hd, n_ctx = 4096, 32, 8, 128, 64
    L = HostLayer(H, nh, nkv, hd, "bf16", layer=5)
    pos = n_ctx
    x = L.x(pos)
    qnw, knw = norm_weights(hd, 5)
    kk0, vv0 = canary(n_ctx, L.nkt, "f16", 31), canary(n_ctx, L.nkt, "f16", 32)
    plan = make_plan(L, "f16", n_ctx, "bf16", theta=THETA)
    Q.qkv_check_device_error()  # clear
    (got,) = run_qknorm(L, plan, x, qnw, knw, pos, kk0, vv0, workspace(plan))
    want = oracle_qknorm(orc, L, x, qnw, knw, pos, kk0, vv0)
    assert want[0] == 1
    compare(L, got, want, pos, "qknorm out of range")
    flags, bad = Q.qkv_check_device_error()
    assert flags & 1 and bad == pos


def _graph_layers(H, nh, nkv, hd, n_layers, n_ctx, pos, mixed=()):
    import torch
    plan_c = Q.qkv_plan_create(H, nh, nkv, hd, THETA, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16)
    plan_m = Q.qkv_plan_create(H, nh, nkv, hd, THETA, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16,
                               layer_class=Q.QKV_CLASS_MIXED)
    layers, plans, host, qn, kn = [], [], [], [], []
    for l in range(n_layers):
        L = HostLayer(H, nh, nkv, hd, "bf16", layer=40 + l)
        dW, db = to_dev(L.W), to_dev(L.bias)
        out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
        dk = torch.zeros(n_ctx, L.nkt, dtype=torch.int16, device="cuda")
        dv = torch.zeros_like(dk)
        a, b = L.nqt, L.nqt + L.nkt
        d = dict(x=to_dev(L.x(pos)), q=out[:a], k=out[a:b], v=out[b:], kv_k=dk, kv_v=dv)
        if l in mixed:
            d.update(wq=dW[:a], wk=dW[a:b], wv=dW[b:], bias_q=db[:a], bias_k=db[a:b], bias_v=db[b:])
            plans.append(plan_m)
        else:
            d.update(w=dW, bias=db)
            plans.append(plan_c)
        qnw, knw = norm_weights(hd, 40 + l)
        layers.append(d)
        host.append((L, qnw, knw, dW, db))
        qn.append(to_dev(qnw))
        kn.append(to_dev(knw))
    return plan_c, plans, layers, host, qn, kn


def test_qknorm_graph_equals_steps_bitwise(qkv):
    """Four Qwen3-14B-shape layers (two concat, two mixed): the graph, replayed twice, equals
    four qkv_decode_step_qknorm calls bit for bit (mixed layers against their concat twins)."""
    import torch
    H, nh, nkv, hd, n_ctx, pos = 5120, 40, 8, 128, 256, 100
    plan_c, plans, layers, host, qn, kn = _graph_layers(H, nh, nkv, hd, 4, n_ctx, pos, mixed=(1, 3))
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    ws = workspace(plan_c)
    stream = torch.cuda.Stream()
    g = Q.qkv_model_graph_create_qknorm(plans, layers, qn, kn, EPS, dpos, ws, stream)
    assert g.kernel_count == 4
    for _ in range(2):
        g.launch(stream)
    stream.synchronize()
    assert not to_host(ws).any()
    for (L, qnw, knw, dW, db), d, dq, dk_w in zip(host, layers, qn, kn):
        out = torch.empty(L.R, dtype=torch.float32, device="cuda")
        dk = torch.zeros(n_ctx, L.nkt, dtype=torch.int16, device="cuda")
        dv = torch.zeros_like(dk)
        a, b = L.nqt, L.nqt + L.nkt
        Q.qkv_decode_step_qknorm(plan_c, d["x"], dW, db, dq, dk_w, EPS, dpos, out[:a], out[a:b], out[b:], dk, dv,
                                 ws, stream=stream)
        stream.synchronize()
        got = torch.cat([d["q"], d["k"], d["v"]])
        assert torch.equal(got.view(torch.int32), out.view(torch.int32))
        assert torch.equal(d["kv_k"], dk) and torch.equal(d["kv_v"], dv)


def test_qknorm_qwen3_14b_48_layer_graph(orc, qkv):
    """The 48-layer Qwen3-14B-shape graph (the workload the bench times), one replay: every
    layer's q, k, v and cache row against the oracle."""
    import torch
    H, nh, nkv, hd, n_ctx, pos = 5120, 40, 8, 128, 4096, 3254
    plan_c, plans, layers, host, qn, kn = _graph_layers(H, nh, nkv, hd, 48, n_ctx, pos)
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    ws = workspace(plan_c)
    stream = torch.cuda.Stream()
    g = Q.qkv_model_graph_create_qknorm(plans, layers, qn, kn, EPS, dpos, ws, stream)
    assert g.kernel_count == 48
    g.launch(stream)
    stream.synchronize()
    assert Q.qkv_check_device_error(stream)[0] == 0
    zero = np.zeros((n_ctx, nkv * hd), np.uint16)
    for l, ((L, qnw, knw, _, _), d) in enumerate(zip(host, layers)):
        st, o, kk, vv = oracle_qknorm(orc, L, to_host(d["x"]), qnw, knw, pos, zero, zero)
        assert st == 0
        got = to_host(torch.cat([d["q"], d["k"], d["v"]]))
        assert_f32_close(got, o, "layer %d q|k|v" % l)
        a, b = L.nqt, L.nqt + L.nkt
        assert_kv_region(to_host(d["kv_k"], np.uint16), kk, pos, "layer %d K" % l, section_f32=o[a:b])
        assert_kv_region(to_host(d["kv_v"], np.uint16), vv, pos, "layer %d V" % l, section_f32=o[b:])
