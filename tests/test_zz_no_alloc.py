"""The allocation-free FusedQkvNorm entry point, qkv_decode_step_qknorm_noalloc.

Some callers cannot allocate device memory at the point where they run the stage: code
inside an allocator or memory-pool callback (allocating there would re-enter the pool),
or a process whose device memory is entirely owned by another framework.  For them the
library keeps the per-head counters in a fixed array of its own, so the call allocates
nothing.  This file is collected last, so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import HostLayer, assert_f32_close, assert_kv_region, canary, to_dev, to_host
from qkv_rope_kv_gb300 import synth

EPS = 1e-6
THETA = 1e6


def test_noalloc_rejects_too_many_heads():
    """More than 1024 q + kv heads cannot fit the fixed array: a clear error, before any CUDA call."""
    lib = Q.load()
    plan = Q.qkv_plan_create(64, 1020, 10, 2, 1e4, 4)
    fake = 16 * 64
    st = lib.qkv_decode_step_qknorm_noalloc(plan.handle, fake, fake, fake, fake, fake, ctypes.c_float(EPS), fake,
                                            fake, fake, fake, fake, fake, None)
    assert st == Q.QKV_ERR_INVALID_ARG
    assert b"1024" in lib.qkv_last_error()


def test_noalloc_accepts_exactly_1024_heads():
    """A plan of exactly 1024 q + kv heads passes the size check: with x null the call fails on
    the null pointer instead, still before any CUDA call (so no device is touched)."""
    lib = Q.load()
    fake = 16 * 64
    for nh, nkv, limit_hit in ((1020, 4, False), (1021, 4, True)):
        plan = Q.qkv_plan_create(64, nh, nkv, 2, 1e4, 4)
        st = lib.qkv_decode_step_qknorm_noalloc(plan.handle, None, fake, fake, fake, fake, ctypes.c_float(EPS),
                                                fake, fake, fake, fake, fake, fake, None)
        assert st == Q.QKV_ERR_INVALID_ARG
        msg = lib.qkv_last_error()
        assert (b"1024" in msg) == limit_hit and (b"x is null" in msg) != limit_hit, msg


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice(qkv):
    """Two calls in a row of the allocation-free entry point, each against the workspace entry
    point on the same inputs (Qwen3-8B layer shape, bf16 weights, f16 cache)."""
    import torch
    H, nh, nkv, hd, n_ctx, pos = 4096, 32, 8, 128, 512, 301
    L = HostLayer(H, nh, nkv, hd, "bf16", layer=7)
    qnw, knw = synth.qk_norm_weights(0, 7, hd)
    plan = Q.qkv_plan_create(H, nh, nkv, hd, THETA, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16)
    dW, db = to_dev(L.W), to_dev(L.bias)
    dq, dk_w = to_dev(qnw), to_dev(knw)
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    kk0, vv0 = canary(n_ctx, L.nkt, "f16", 41), canary(n_ctx, L.nkt, "f16", 42)
    a, b = L.nqt, L.nqt + L.nkt

    def run(fn, x):
        out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
        dk, dv = to_dev(kk0), to_dev(vv0)
        fn(to_dev(x), out, dk, dv)
        torch.cuda.synchronize()
        return to_host(out), to_host(dk, np.uint16), to_host(dv, np.uint16)

    ws = torch.zeros(Q.qkv_qknorm_workspace_bytes(plan) // 4, dtype=torch.int32, device="cuda")
    for call, xpos in enumerate((pos, pos + 1)):
        x = L.x(xpos)
        want = run(lambda dx, o, dk, dv: Q.qkv_decode_step_qknorm(plan, dx, dW, db, dq, dk_w, EPS, dpos, o[:a],
                                                                  o[a:b], o[b:], dk, dv, ws), x)
        got = run(lambda dx, o, dk, dv: Q.qkv_decode_step_qknorm_noalloc(plan, dx, dW, db, dq, dk_w, EPS, dpos,
                                                                         o[:a], o[a:b], o[b:], dk, dv), x)
        assert_f32_close(got[0], want[0], "call %d q|k|v" % call)
        assert_kv_region(got[1], want[1], pos, "call %d K" % call, section_f32=want[0][a:b])
        assert_kv_region(got[2], want[2], pos, "call %d V" % call, section_f32=want[0][b:])
    assert Q.qkv_check_device_error()[0] == 0


@pytest.mark.gpu
def test_noalloc_at_the_head_limit_matches_oracle(orc, qkv):
    """A plan of exactly 1024 q + kv heads (1020 q, 4 kv, head_dim 2, hidden 64, bf16 weights,
    f16 cache) through the allocation-free entry point, against the oracle's FusedQkvNorm."""
    import torch
    H, nh, nkv, hd, n_ctx, pos = 64, 1020, 4, 2, 8, 5
    L = HostLayer(H, nh, nkv, hd, "bf16", layer=9)
    qnw, knw = synth.qk_norm_weights(0, 9, hd)
    plan = Q.qkv_plan_create(H, nh, nkv, hd, THETA, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16)
    kk0, vv0 = canary(n_ctx, L.nkt, "f16", 51), canary(n_ctx, L.nkt, "f16", 52)
    x = L.x(pos)
    out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
    dk, dv = to_dev(kk0), to_dev(vv0)
    a, b = L.nqt, L.nqt + L.nkt
    Q.qkv_decode_step_qknorm_noalloc(plan, to_dev(x), to_dev(L.W), to_dev(L.bias), to_dev(qnw), to_dev(knw), EPS,
                                     torch.tensor([pos], dtype=torch.int32, device="cuda"), out[:a], out[a:b],
                                     out[b:], dk, dv)
    torch.cuda.synchronize()
    kk, vv = kk0.copy(), vv0.copy()
    st, q, k, v = orc.decode_qknorm(L.W, x, L.bias, qnw, knw, EPS, nh, nkv, hd, THETA, 1.0, pos, kk, vv)
    assert st == 0
    got = to_host(out)
    assert_f32_close(got[:a], q, "1024 heads q")
    assert_f32_close(got[a:b], k, "1024 heads k")
    assert_f32_close(got[b:], v, "1024 heads v")
    assert_kv_region(to_host(dk, np.uint16), kk, pos, "1024 heads K", section_f32=k)
    assert_kv_region(to_host(dv, np.uint16), vv, pos, "1024 heads V", section_f32=v)
    assert Q.qkv_check_device_error()[0] == 0


@pytest.mark.gpu
def test_noalloc_after_out_of_range_position(orc, qkv):
    """A call with a position past the cache sets the device flag and stores nothing; once the
    flag is read (and so cleared) the next call, on the same shared counters, matches the
    oracle."""
    import torch
    H, nh, nkv, hd, n_ctx = 1024, 8, 2, 64, 16
    L = HostLayer(H, nh, nkv, hd, "bf16", layer=10)
    qnw, knw = synth.qk_norm_weights(0, 10, hd)
    plan = Q.qkv_plan_create(H, nh, nkv, hd, THETA, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16)
    kk0, vv0 = canary(n_ctx, L.nkt, "f16", 61), canary(n_ctx, L.nkt, "f16", 62)
    dW, db, dq, dkn = to_dev(L.W), to_dev(L.bias), to_dev(qnw), to_dev(knw)
    dk, dv = to_dev(kk0), to_dev(vv0)
    a, b = L.nqt, L.nqt + L.nkt
    Q.qkv_check_device_error()
    for pos, bad in ((n_ctx + 3, True), (11, False)):
        out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
        Q.qkv_decode_step_qknorm_noalloc(plan, to_dev(L.x(pos)), dW, db, dq, dkn, EPS,
                                         torch.tensor([pos], dtype=torch.int32, device="cuda"), out[:a], out[a:b],
                                         out[b:], dk, dv)
        torch.cuda.synchronize()
        flags, bad_pos = Q.qkv_check_device_error()
        kk, vv = kk0.copy(), vv0.copy()
        st, q, k, v = orc.decode_qknorm(L.W, L.x(pos), L.bias, qnw, knw, EPS, nh, nkv, hd, THETA, 1.0, pos, kk, vv)
        got = to_host(out)
        assert_f32_close(got, np.concatenate([q, k, v]), "pos %d q|k|v" % pos)
        if bad:
            assert flags & 1 and bad_pos == pos and st == 1
            assert_kv_region(to_host(dk, np.uint16), kk0, None, "pos %d K" % pos)
            assert_kv_region(to_host(dv, np.uint16), vv0, None, "pos %d V" % pos)
        else:
            assert flags == 0 and st == 0
            assert_kv_region(to_host(dk, np.uint16), kk, pos, "pos %d K" % pos, section_f32=k)
            assert_kv_region(to_host(dv, np.uint16), vv, pos, "pos %d V" % pos, section_f32=v)
