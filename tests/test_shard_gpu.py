"""Head sharding on the CUDA path, on one GPU: for each rank of W, a plan of that rank's heads
(shard.head_shard) runs qkv_decode_step on its rows of W and bias into its own
[n_ctx x nkt/W] cache regions; gathered, the ranks' q|k|v and cache columns equal the
unsharded plan's bit for bit.  Every row is reduced by the same code whatever the number of
rows (the reduction order depends only on H), and the epilogue of a row depends only on its
position inside its head, so the split needs no exchange step."""
import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import HostLayer, canary, to_dev, to_host
from qkv_rope_kv_gb300 import shard

pytestmark = pytest.mark.gpu

CASES = [
    # H, nh, nkv, hd, world, layer class
    (5120, 40, 8, 128, 2, Q.QKV_CLASS_CONCAT),
    (5120, 40, 8, 128, 4, Q.QKV_CLASS_CONCAT),
    (5120, 40, 8, 128, 8, Q.QKV_CLASS_CONCAT),
    (5120, 40, 8, 128, 2, Q.QKV_CLASS_MIXED),
    (3584, 28, 4, 128, 2, Q.QKV_CLASS_CONCAT),
    (3584, 28, 4, 128, 4, Q.QKV_CLASS_CONCAT),
]


def run_plan(L_W, L_b, nh, nkv, hd, H, x, pos, kk0, vv0, cls, n_ctx):
    import torch
    plan = Q.qkv_plan_create(H, nh, nkv, hd, 1e6, n_ctx, w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16, layer_class=cls)
    nqt, nkt = nh * hd, nkv * hd
    out = torch.full((nqt + 2 * nkt,), float("nan"), dtype=torch.float32, device="cuda")
    dk, dv = to_dev(kk0), to_dev(vv0)
    dW, db = to_dev(L_W), to_dev(L_b)
    dpos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    q, k, v = out[:nqt], out[nqt:nqt + nkt], out[nqt + nkt:]
    if cls == Q.QKV_CLASS_CONCAT:
        Q.qkv_decode_step(plan, to_dev(x), dW, db, dpos, q, k, v, dk, dv)
    else:
        a, b = nqt, nqt + nkt
        Q.qkv_decode_step_mixed(plan, to_dev(x), dW[:a].contiguous(), dW[a:b].contiguous(), dW[b:].contiguous(),
                                db[:a], db[a:b], db[b:], dpos, q, k, v, dk, dv)
    torch.cuda.synchronize()
    assert Q.qkv_check_device_error()[0] == 0
    return to_host(out), to_host(dk, np.uint16), to_host(dv, np.uint16)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "H%d_kv%d_world%d_%s" % (c[0], c[2], c[4],
                                                                                 "concat" if c[5] == 0 else "mixed"))
def test_sharded_plans_equal_unsharded_bitwise(qkv, case):
    H, nh, nkv, hd, world, cls = case
    n_ctx, pos = 48, 37
    L = HostLayer(H, nh, nkv, hd, "bf16", layer=21)
    x = L.x(pos)
    kk0, vv0 = canary(n_ctx, L.nkt, "f16", 81), canary(n_ctx, L.nkt, "f16", 82)
    full = run_plan(L.W, L.bias, nh, nkv, hd, H, x, pos, kk0, vv0, cls, n_ctx)
    got_out = np.full(L.R, np.nan, np.float32)
    got_k = np.zeros_like(kk0)
    got_v = np.zeros_like(vv0)
    for r in range(world):
        s = shard.head_shard(nh, nkv, hd, world, r)
        rows = np.concatenate([np.arange(a, b) for a, b in s.concat_rows])
        c0, c1 = s.kv_cols
        out, dk, dv = run_plan(np.ascontiguousarray(L.W[rows]), np.ascontiguousarray(L.bias[rows]), s.n_head,
                               s.n_head_kv, hd, H, x, pos, np.ascontiguousarray(kk0[:, c0:c1]),
                               np.ascontiguousarray(vv0[:, c0:c1]), cls, n_ctx)
        got_out[rows] = out
        got_k[:, c0:c1] = dk
        got_v[:, c0:c1] = dv
    assert np.array_equal(got_out.view(np.uint32), full[0].view(np.uint32))
    assert np.array_equal(got_k, full[1]) and np.array_equal(got_v, full[2])
