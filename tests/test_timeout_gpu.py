"""The device-side failure path of the decode rings, made to happen without a GPU fault.

Every wait of a ring kernel on a pipeline barrier is bounded.  The test hook
qkv_test_decode_wait_timeout (include/qkv_test.h) withholds the last weight copy of
every CTA and limits each wait to 200 us, so the consumer waiting for that copy gives
up: the launch must still complete, the device status word must carry the timeout
flag (2), no cache row other than the step's position may change, and the next
ordinary call on the same context must match the oracle.  Shapes cover the three ring
shapes: the block ring (rows of 8 KB), the pair ring (4-8 KB rows) and the short-row
pair ring (rows under 4 KB, f32 weights).
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
