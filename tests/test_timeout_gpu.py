"""The device-side failure paths of the decode rings and of the prefill, made to happen
without a GPU fault.

Every wait of a ring kernel on a pipeline barrier is bounded.  The test hook
qkv_test_decode_wait_timeout (include/qkv_test.h) withholds the last weight copy of
every CTA and limits each wait to 200 us, so the consumer waiting for that copy gives
up: the launch must still complete, the device status word must carry the timeout
flag (2), no cache row other than the step's position may change, and the next
ordinary call on the same context must match the oracle.  Shapes cover the three ring
shapes: the block ring (rows of 8 KB), the pair ring (4-8 KB rows) and the short-row
pair ring (rows under 4 KB, f32 weights).

qkv_test_prefill_xchg_timeout withholds the prefill's exchange of partial sums between
the two CTAs of each cluster (the two K halves of a 128-row block), so every CTA's wait
for its peer's partial runs out: the flag must be set, no Y row and no cache row may be
written, and the next ordinary prefill must match the oracle.
"""
import time

import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import HostLayer, assert_f32_close, assert_kv_region, canary, to_dev, to_host

pytestmark = pytest.mark.gpu

SHAPES = [
    # H, nh, nkv, hd, w_dtype: rows of 8 KB (block ring), 4 KB (pair ring), 3.5 KB f32 (short-row ring)
    (4096, 8, 2, 128, "bf16"),
    (2048, 6, 2, 64, "bf16"),
    (896, 14, 2, 64, "f32"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_%s" % (s[0], s[4]))
def test_withheld_copy_times_out_and_context_stays_usable(orc, qkv, shape):
    import torch
    H, nh, nkv, hd, w_dtype = shape
    n_ctx, pos = 16, 9
    L = HostLayer(H, nh, nkv, hd, w_dtype, layer=3)
    plan = Q.qkv_plan_create(H, nh, nkv, hd, 1e6, n_ctx, w_dtype=Q.QKV_BF16 if w_dtype == "bf16" else Q.QKV_F32,
                             kv_dtype=Q.QKV_F16)
    kk0, vv0 = canary(n_ctx, L.nkt, "f16", 71), canary(n_ctx, L.nkt, "f16", 72)
    dW, db, dx = to_dev(L.W), to_dev(L.bias), to_dev(L.x(pos))
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    dk, dv = to_dev(kk0), to_dev(vv0)
    out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
    a, b = L.nqt, L.nqt + L.nkt
    Q.qkv_check_device_error()
    t0 = time.perf_counter()
    Q.qkv_test_decode_wait_timeout(plan, dx, dW, db, dpos, out[:a], out[a:b], out[b:], dk, dv, wait_limit_us=200)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    flags, _ = Q.qkv_check_device_error()
    assert flags & 2, "no timeout flag after a withheld copy (flags %#x)" % flags
    # the failed launch wrote nothing outside row pos of the caches
    keep = np.arange(n_ctx) != pos
    assert np.array_equal(to_host(dk, np.uint16)[keep], kk0[keep])
    assert np.array_equal(to_host(dv, np.uint16)[keep], vv0[keep])

    # the context is usable: an ordinary call on fresh buffers matches the oracle
    dk, dv = to_dev(kk0), to_dev(vv0)
    out = torch.full((L.R,), float("nan"), dtype=torch.float32, device="cuda")
    Q.qkv_decode_step(plan, dx, dW, db, dpos, out[:a], out[a:b], out[b:], dk, dv)
    torch.cuda.synchronize()
    assert Q.qkv_check_device_error()[0] == 0
    kk, vv = kk0.copy(), vv0.copy()
    st, q, k, v = orc.decode(L.W, L.x(pos), L.bias, nh, nkv, hd, 1e6, 1.0, pos, kk, vv)
    got = to_host(out)
    assert_f32_close(got[:a], q, "after timeout q")
    assert_f32_close(got[a:b], k, "after timeout k")
    assert_f32_close(got[b:], v, "after timeout v")
    assert_kv_region(to_host(dk, np.uint16), kk, pos, "after timeout K", section_f32=k)
    assert_kv_region(to_host(dv, np.uint16), vv, pos, "after timeout V", section_f32=v)


PREFILL_SHAPES = [
    # H, nh, nkv, hd, nt, kv dtype: heads of 64 (clusters span two heads), heads of 128 with two token tiles
    (1024, 4, 2, 64, 40, "f16"),
    (640, 2, 1, 128, 130, "f32"),
]


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=lambda s: "H%d_d%d_nt%d_%s" % (s[0], s[3], s[4], s[5]))
def test_prefill_withheld_exchange_times_out_and_context_stays_usable(orc, qkv, shape):
    import torch
    from qkv_rope_kv_gb300 import synth
    from test_prefill_gpu import DT, check, oracle_prefill, run_prefill
    H, nh, nkv, hd, nt, kvdt = shape
    n_ctx = nt + 10
    R = (nh + 2 * nkv) * hd
    W = synth.weight_rows(0, 5, 0, R, H, "bf16")
    b = synth.bias(0, 5, R)
    X = synth.prefill_x(0, 5, nt, H)
    positions = np.random.default_rng(nt + H).permutation(n_ctx)[:nt].astype(np.int32)
    kk0, vv0 = canary(n_ctx, nkv * hd, kvdt, 81), canary(n_ctx, nkv * hd, kvdt, 82)
    plan = Q.qkv_plan_create(H, nh, nkv, hd, 1e6, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=DT[kvdt])
    dY = torch.full((nt, R), float("nan"), dtype=torch.float32, device="cuda")
    dk, dv = to_dev(kk0), to_dev(vv0)
    dpos = torch.from_numpy(positions).cuda()
    Q.qkv_check_device_error()
    t0 = time.perf_counter()
    Q.qkv_test_prefill_xchg_timeout(plan, to_dev(X), nt, to_dev(W), to_dev(b), dpos, dY, dk, dv, wait_limit_us=200)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    flags, _ = Q.qkv_check_device_error()
    assert flags & 2, "no timeout flag after a withheld exchange (flags %#x)" % flags
    # no CTA received its peer's partial: no Y row and no cache row was written
    assert np.isnan(to_host(dY)).all()
    bits = np.uint32 if kvdt == "f32" else np.uint16
    assert np.array_equal(to_host(dk, bits), kk0.view(bits))
    assert np.array_equal(to_host(dv, bits), vv0.view(bits))

    # the context is usable: an ordinary prefill matches the per-token oracle
    got = run_prefill(H, nh, nkv, hd, n_ctx, kvdt, X, W, b, positions, kk0, vv0)
    assert Q.qkv_check_device_error()[0] == 0
    want = oracle_prefill(orc, X, W, b, positions, nh, nkv, hd, kk0, vv0)
    check(nh, nkv, hd, got, want, positions, "prefill after timeout")
