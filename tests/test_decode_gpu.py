"""Decode kernels against the CPU oracle, element by element, through the C ABI.

Covers ragged 16-byte tails, the scalar (unaligned-row) path, tiny heads,
several tiles per SM, both layer classes, f32 and f16 caches, position 0 and
the last cache row, the bitwise gates of the fusion (fused == projection +
one-launch epilogue == projection + seven-launch chain, both pointer forms),
class equivalence, and out-of-range positions (device status, no store).
"""
import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import (HostLayer, assert_f32_close, assert_kv_region, canary, to_dev, to_host)

pytestmark = pytest.mark.gpu

DT = {"f32": Q.QKV_F32, "bf16": Q.QKV_BF16, "f16": Q.QKV_F16}


def kv_np(kv_dtype):
    return np.float32 if kv_dtype == "f32" else np.uint16


def make_plan(L, kv_dtype, n_ctx, w_dtype, cls=Q.QKV_CLASS_CONCAT, theta=1e6):
    return Q.qkv_plan_create(L.H, L.nh, L.nkv, L.hd, theta, n_ctx, w_dtype=DT[w_dtype],
                             kv_dtype=DT[kv_dtype], layer_class=cls)


def run_gpu(L, plan, cls, x, pos, kk0, vv0, w_dev=None):
    import torch
    dW = to_dev(L.W) if w_dev is None else w_dev
    db = to_dev(L.bias)
    dx = to_dev(x)
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    out = torch.empty(L.R, dtype=torch.float32, device="cuda")
    dk, dv = to_dev(kk0), to_dev(vv0)
    q, k, v = out[:L.nqt], out[L.nqt:L.nqt + L.nkt], out[L.nqt + L.nkt:]
    if cls == Q.QKV_CLASS_CONCAT:
        Q.qkv_decode_step(plan, dx, dW, db, dpos, q, k, v, dk, dv)
    else:
        a, b = L.nqt, L.nqt + L.nkt
        Q.qkv_decode_step_mixed(plan, dx, dW[:a].contiguous(), dW[a:b].contiguous(),
                                dW[b:].contiguous(), db[:a], db[a:b], db[b:], dpos, q, k, v, dk, dv)
    torch.cuda.synchronize()
    return to_host(out), to_host(dk, kv_np(plan_kv(plan))), to_host(dv, kv_np(plan_kv(plan)))


def plan_kv(plan):
    return "f32" if plan.desc.kv_dtype == Q.QKV_F32 else "f16"


def oracle_run(orc, L, x, pos, kk0, vv0, theta=1e6):
    kk, vv = kk0.copy(), vv0.copy()
    st, q, k, v = orc.decode(L.W, x, L.bias, L.nh, L.nkv, L.hd, theta, 1.0, pos, kk, vv)
    return st, np.concatenate([q, k, v]), kk, vv


def compare(L, got, want, pos, what):
    out, kk, vv = got
    st, o_out, o_kk, o_vv = want
    assert_f32_close(out[:L.nqt], o_out[:L.nqt], what + " q")
    assert_f32_close(out[L.nqt:L.nqt + L.nkt], o_out[L.nqt:L.nqt + L.nkt], what + " k")
    assert_f32_close(out[L.nqt + L.nkt:], o_out[L.nqt + L.nkt:], what + " v")
    in_range = st == 0
    assert_kv_region(kk, o_kk, pos if in_range else None, what + " K",
                     section_f32=o_out[L.nqt:L.nqt + L.nkt])
    assert_kv_region(vv, o_vv, pos if in_range else None, what + " V",
                     section_f32=o_out[L.nqt + L.nkt:])


SHAPES = [
    # H, nh, nkv, hd, w_dtype, kv_dtype, n_ctx, pos
    (1000, 6, 2, 64, "bf16", "f16", 37, 29),   # 125 chunks per row: ragged tail of the unrolled loop
    (1000, 6, 2, 64, "f32", "f32", 37, 0),     # position 0: rotation is the identity
    (1001, 3, 1, 32, "bf16", "f32", 8, 7),     # rows not 16-byte aligned: scalar path; last cache row
    (1002, 3, 1, 32, "f32", "f16", 8, 5),      # f32 rows of 4008 bytes: scalar path
    (40, 3, 1, 8, "f32", "f16", 5, 3),
    (8, 1, 1, 2, "bf16", "f16", 2, 1),         # hd = 2: one pair per head
    (4104, 7, 3, 128, "bf16", "f16", 300, 257),
    (896, 14, 2, 64, "f32", "f32", 512, 17),   # Qwen2.5-0.5B single layer
    (3584, 28, 4, 128, "bf16", "f16", 4096, 1641),  # Qwen2.5-7B layer
    (5120, 40, 8, 128, "bf16", "f16", 4096, 3254),  # Qwen2.5-14B layer
    (256, 64, 8, 128, "bf16", "f16", 64, 33),  # 5120 row pairs, 16-stage ring wraps twice per CTA
    (1024, 96, 16, 64, "f32", "f32", 40, 39),  # f32 rows, 4 KB stages, ring wraps per CTA
    (2048, 8, 2, 128, "f32", "f16", 64, 20),   # f32 rows of 8 KB: block ring
    (4096, 64, 8, 128, "bf16", "f32", 16, 15),  # block ring wraps several times per CTA
    (4096, 3, 1, 2, "bf16", "f16", 4, 2),      # hd = 2: single-row blocks
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_h%d_kv%d_d%d_%s_%s" % s[:6])
@pytest.mark.parametrize("cls", [Q.QKV_CLASS_CONCAT, Q.QKV_CLASS_MIXED], ids=["concat", "mixed"])
def test_decode_matches_oracle(orc, qkv, shape, cls):
    H, nh, nkv, hd, wdt, kvdt, n_ctx, pos = shape
    L = HostLayer(H, nh, nkv, hd, wdt, layer=3)
    x = L.x(pos)
    kk0, vv0 = canary(n_ctx, L.nkt, kvdt, 1), canary(n_ctx, L.nkt, kvdt, 2)
    plan = make_plan(L, kvdt, n_ctx, wdt, cls)
    got = run_gpu(L, plan, cls, x, pos, kk0, vv0)
    want = oracle_run(orc, L, x, pos, kk0, vv0)
    assert want[0] == 0
    compare(L, got, want, pos, "decode %s" % (shape,))


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[8]], ids=["small", "7b"])
def test_concat_equals_mixed_bitwise(qkv, shape):
    """Rows are reduced independently, so the concat class and the same rows in
    three matrices give identical bits ("73 · D3-8", §2, concat matmul)."""
    H, nh, nkv, hd, wdt, kvdt, n_ctx, pos = shape
    L = HostLayer(H, nh, nkv, hd, wdt, layer=5)
    x = L.x(pos)
    kk0, vv0 = canary(n_ctx, L.nkt, kvdt, 3), canary(n_ctx, L.nkt, kvdt, 4)
    a = run_gpu(L, make_plan(L, kvdt, n_ctx, wdt, Q.QKV_CLASS_CONCAT), Q.QKV_CLASS_CONCAT, x, pos, kk0, vv0)
    b = run_gpu(L, make_plan(L, kvdt, n_ctx, wdt, Q.QKV_CLASS_MIXED), Q.QKV_CLASS_MIXED, x, pos, kk0, vv0)
    for u, w in zip(a, b):
        assert np.array_equal(u.view(np.uint8), w.view(np.uint8))


@pytest.mark.parametrize("shape", [SHAPES[8], SHAPES[9], SHAPES[3]], ids=["7b", "14b", "small_f32kv"])
@pytest.mark.parametrize("kvdt", ["f32", "f16"])
def test_fused_equals_epilogue_equals_chain_bitwise(qkv, shape, kvdt):
    """The page's bitwise gate: one fused launch == projection + one-launch
    epilogue (both pointer forms) == projection + the seven-launch chain."""
    import torch
    H, nh, nkv, hd, wdt, _, n_ctx, pos = shape
    L = HostLayer(H, nh, nkv, hd, wdt, layer=7)
    x = L.x(pos)
    kk0, vv0 = canary(n_ctx, L.nkt, kvdt, 5), canary(n_ctx, L.nkt, kvdt, 6)
    plan = make_plan(L, kvdt, n_ctx, wdt)
    fused = run_gpu(L, plan, Q.QKV_CLASS_CONCAT, x, pos, kk0, vv0)

    dW, db, dx = to_dev(L.W), to_dev(L.bias), to_dev(x)
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    a, b = L.nqt, L.nqt + L.nkt
    wq, wk, wv = dW[:a], dW[a:b], dW[b:]
    bq, bk, bv = db[:a], db[a:b], db[b:]

    # form 1: sections of one concat output buffer
    y1 = torch.empty(L.R, dtype=torch.float32, device="cuda")
    dk1, dv1 = to_dev(kk0), to_dev(vv0)
    Q.qkv_project(plan, dx, wq, wk, wv, y1[:a], y1[a:b], y1[b:])
    Q.qkv_epilogue(plan, y1[:a], y1[a:b], y1[b:], bq, bk, bv, dpos, dk1, dv1)
    # form 2: three separate buffers
    q2 = torch.empty(L.nqt, dtype=torch.float32, device="cuda")
    k2 = torch.empty(L.nkt, dtype=torch.float32, device="cuda")
    v2 = torch.empty(L.nkt, dtype=torch.float32, device="cuda")
    dk2, dv2 = to_dev(kk0), to_dev(vv0)
    Q.qkv_project(plan, dx, wq, wk, wv, q2, k2, v2)
    Q.qkv_epilogue(plan, q2, k2, v2, bq, bk, bv, dpos, dk2, dv2)
    # the unfused chain: bias x3, rope x2, store x2
    y3 = torch.empty(L.R, dtype=torch.float32, device="cuda")
    dk3, dv3 = to_dev(kk0), to_dev(vv0)
    Q.qkv_project(plan, dx, wq, wk, wv, y3[:a], y3[a:b], y3[b:])
    Q.qkv_chain_add_bias(y3[:a], bq, L.nqt)
    Q.qkv_chain_add_bias(y3[a:b], bk, L.nkt)
    Q.qkv_chain_add_bias(y3[b:], bv, L.nkt)
    Q.qkv_chain_rope(plan, y3[:a], L.nh, dpos)
    Q.qkv_chain_rope(plan, y3[a:b], L.nkv, dpos)
    Q.qkv_chain_store(plan, y3[a:b], dk3, dpos)
    Q.qkv_chain_store(plan, y3[b:], dv3, dpos)
    torch.cuda.synchronize()

    kvt = kv_np(kvdt)
    forms = [
        (to_host(y1), to_host(dk1, kvt), to_host(dv1, kvt)),
        (np.concatenate([to_host(q2), to_host(k2), to_host(v2)]), to_host(dk2, kvt), to_host(dv2, kvt)),
        (to_host(y3), to_host(dk3, kvt), to_host(dv3, kvt)),
    ]
    for i, f in enumerate(forms):
        for u, w in zip(fused, f):
            assert np.array_equal(u.view(np.uint8), w.view(np.uint8)), "form %d differs" % i


@pytest.mark.parametrize("bad_pos", [-1, 12, 4000])
def test_out_of_range_position_sets_flag_and_skips_store(orc, qkv, bad_pos):
    H, nh, nkv, hd, n_ctx = 256, 4, 2, 16, 12
    L = HostLayer(H, nh, nkv, hd, "bf16", layer=1)
    x = L.x(5)
    kk0, vv0 = canary(n_ctx, L.nkt, "f16", 7), canary(n_ctx, L.nkt, "f16", 8)
    Q.qkv_check_device_error()  # clear anything left over
    plan = make_plan(L, "f16", n_ctx, "bf16")
    got = run_gpu(L, plan, Q.QKV_CLASS_CONCAT, x, bad_pos, kk0, vv0)
    flags, where = Q.qkv_check_device_error()
    assert flags & 1 and where == bad_pos
    assert Q.qkv_check_device_error()[0] == 0  # reading cleared it
    want = oracle_run(orc, L, x, bad_pos, kk0, vv0)
    assert want[0] == 1  # the oracle reports the range error too
    compare(L, got, want, bad_pos, "bad pos %d" % bad_pos)
    with pytest.raises(Q.QkvError):
        got = run_gpu(L, plan, Q.QKV_CLASS_CONCAT, x, bad_pos, kk0, vv0)
        Q.qkv_check_device_error(raise_on_flag=True)


def test_repeated_steps_fill_consecutive_rows(orc, qkv):
    """A decode loop: positions 0..5 land in rows 0..5; later rows keep their canary."""
    import torch
    H, nh, nkv, hd, n_ctx = 512, 4, 2, 32, 9
    L = HostLayer(H, nh, nkv, hd, "bf16", layer=2)
    plan = make_plan(L, "f16", n_ctx, "bf16")
    kk, vv = canary(n_ctx, L.nkt, "f16", 9), canary(n_ctx, L.nkt, "f16", 10)
    ok, ov = kk.copy(), vv.copy()
    dW, db = to_dev(L.W), to_dev(L.bias)
    dk, dv = to_dev(kk), to_dev(vv)
    out = torch.empty(L.R, dtype=torch.float32, device="cuda")
    for pos in range(6):
        x = L.x(pos)
        dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
        Q.qkv_decode_step(plan, to_dev(x), dW, db, dpos, out[:L.nqt], out[L.nqt:L.nqt + L.nkt],
                          out[L.nqt + L.nkt:], dk, dv)
        st, q, k, v = orc.decode(L.W, x, L.bias, nh, nkv, hd, 1e6, 1.0, pos, ok, ov)
        torch.cuda.synchronize()
        assert_f32_close(to_host(out), np.concatenate([q, k, v]), "step %d" % pos)
    assert_kv_region(to_host(dk, np.uint16), ok, list(range(6)), "K")
    assert_kv_region(to_host(dv, np.uint16), ov, list(range(6)), "V")
