"""The RMSNorm prologue fused into the decode projection, against the oracle:
oracle RMSNorm of h (plain definition; the pages name the op only), then the oracle
stage on that x.  Shapes reach the block ring (rows >= 8 KB), the pair ring and the
register-streaming kernel (unaligned rows); the normed graph (both layer classes)
against sequential normed steps, bitwise."""
import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import HostLayer, canary, to_dev, to_host
from qkv_rope_kv_gb300 import synth
from test_decode_gpu import compare, kv_np, make_plan, oracle_run

pytestmark = pytest.mark.gpu

EPS = 1e-6

SHAPES = [
    # H, nh, nkv, hd, w dtype, kv dtype, n_ctx, pos
    (5120, 40, 8, 128, "bf16", "f16", 4096, 3254),  # 14B layer: block ring
    (4104, 7, 3, 128, "bf16", "f16", 300, 257),      # block ring, ragged heads
    (3584, 28, 4, 128, "bf16", "f16", 4096, 1641),   # 7B layer: pair ring
    (896, 14, 2, 64, "f32", "f32", 512, 17),         # 0.5B layer: pair ring, f32 rows
    (1001, 3, 1, 32, "bf16", "f32", 8, 7),           # unaligned rows: register kernel
    (1002, 3, 1, 32, "f32", "f16", 8, 5),            # unaligned f32 rows: register kernel
]


def run_normed(L, plan, h, nw, pos, kk0, vv0):
    import torch
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    out = torch.empty(L.R, dtype=torch.float32, device="cuda")
    dk, dv = to_dev(kk0), to_dev(vv0)
    q, k, v = out[:L.nqt], out[L.nqt:L.nqt + L.nkt], out[L.nqt + L.nkt:]
    Q.qkv_decode_step_rmsnorm(plan, to_dev(h), to_dev(nw), EPS, to_dev(L.W), to_dev(L.bias), dpos, q, k, v, dk, dv)
    torch.cuda.synchronize()
    kvt = kv_np("f32" if plan.desc.kv_dtype == Q.QKV_F32 else "f16")
    return to_host(out), to_host(dk, kvt), to_host(dv, kvt)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_h%d_kv%d_d%d_%s_%s" % s[:6])
def test_rmsnorm_decode_matches_oracle(orc, qkv, shape):
    H, nh, nkv, hd, wdt, kvdt, n_ctx, pos = shape
    L = HostLayer(H, nh, nkv, hd, wdt, layer=4)
    h = (np.float32(3.0) * L.x(pos)).astype(np.float32)  # not unit RMS: the norm matters
    nw = synth.norm_weight(0, 4, H)
    kk0, vv0 = canary(n_ctx, L.nkt, kvdt, 11), canary(n_ctx, L.nkt, kvdt, 12)
    got = run_normed(L, make_plan(L, kvdt, n_ctx, wdt), h, nw, pos, kk0, vv0)
    want = oracle_run(orc, L, orc.rmsnorm(h, nw, EPS), pos, kk0, vv0)
    assert want[0] == 0
    compare(L, got, want, pos, "rmsnorm decode %s" % (shape,))


def test_rmsnorm_graph_equals_steps_bitwise(qkv):
    """Four layers (two concat, two mixed) of the 14B shape: the normed graph, replayed twice,
    == four qkv_decode_step_rmsnorm / mixed-class steps on the same inputs (concat only has a
    direct entry point, so the mixed layers are compared with their concat twins)."""
    import torch
    H, nh, nkv, hd = 5120, 40, 8, 128
    n_ctx, pos = 256, 100
    plan_c = Q.qkv_plan_create(H, nh, nkv, hd, 1e6, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16)
    plan_m = Q.qkv_plan_create(H, nh, nkv, hd, 1e6, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16,
                               layer_class=Q.QKV_CLASS_MIXED)
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    layers, norms, plans, step_args = [], [], [], []
    for l in range(4):
        L = HostLayer(H, nh, nkv, hd, "bf16", layer=20 + l)
        dW, db = to_dev(L.W), to_dev(L.bias)
        dh = to_dev((np.float32(0.5) * L.x(pos)).astype(np.float32))
        dn = to_dev(synth.norm_weight(0, 20 + l, H))
        out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
        dk = torch.zeros(n_ctx, L.nkt, dtype=torch.int16, device="cuda")
        dv = torch.zeros_like(dk)
        a, b = L.nqt, L.nqt + L.nkt
        d = dict(x=dh, q=out[:a], k=out[a:b], v=out[b:], kv_k=dk, kv_v=dv)
        if l % 2:
            d.update(wq=dW[:a], wk=dW[a:b], wv=dW[b:], bias_q=db[:a], bias_k=db[a:b], bias_v=db[b:])
            plans.append(plan_m)
        else:
            d.update(w=dW, bias=db)
            plans.append(plan_c)
        layers.append(d)
        norms.append(dn)
        step_args.append((dh, dn, dW, db, L))
    stream = torch.cuda.Stream()
    g = Q.qkv_model_graph_create_rmsnorm(plans, layers, norms, EPS, dpos, stream)
    assert g.kernel_count == 4
    for _ in range(2):
        g.launch(stream)
    stream.synchronize()
    for (dh, dn, dW, db, L), d in zip(step_args, layers):
        out = torch.empty(L.R, dtype=torch.float32, device="cuda")
        dk = torch.zeros(n_ctx, L.nkt, dtype=torch.int16, device="cuda")
        dv = torch.zeros_like(dk)
        a, b = L.nqt, L.nqt + L.nkt
        Q.qkv_decode_step_rmsnorm(plan_c, dh, dn, EPS, dW, db, dpos, out[:a], out[a:b], out[b:], dk, dv,
                                  stream=stream)
        stream.synchronize()
        got = torch.cat([d["q"], d["k"], d["v"]])
        assert torch.equal(got.view(torch.int32), out.view(torch.int32))
        assert torch.equal(d["kv_k"], dk) and torch.equal(d["kv_v"], dv)
