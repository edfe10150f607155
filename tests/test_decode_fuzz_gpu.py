"""Seeded random decode shapes against the CPU oracle, element by element.

The hand-picked shapes of test_decode_gpu.py cover each kernel path at its edges; these
cover the combinations between them: row widths on both sides of the ring thresholds
(4 KB and 8 KB rows) and far past them, mostly 16-byte aligned rows with some that are not
(the register-streaming path), head widths from 2 to 256, q head counts that are any
multiple of the kv head count, both weight and cache types, both layer classes, and a
random position in a short cache.  The generator is seeded, so every run sees the same
shapes.
"""
import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import HostLayer, canary
from test_decode_gpu import compare, make_plan, oracle_run, run_gpu

pytestmark = pytest.mark.gpu

CLASSES = (Q.QKV_CLASS_CONCAT, Q.QKV_CLASS_MIXED)


def fuzz_shapes(n=24, seed=20261202, max_weight_bytes=48 << 20):
    """(H, nh, nkv, hd, w dtype, kv dtype, n_ctx, pos, class) tuples."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        wdt = ("f32", "bf16")[int(rng.integers(2))]
        es = 4 if wdt == "f32" else 2
        row_bytes = int(rng.choice([1024, 3000, 4096, 6000, 8192, 10240, 12288]))
        H = max(8, row_bytes // es + int(rng.integers(-40, 41)))
        if rng.random() < 0.75:
            H -= H % (16 // es)  # a 16-byte aligned row
        hd = 2 * int(rng.integers(1, 129))
        nkv = int(rng.integers(1, 5))
        nh = nkv * int(rng.integers(1, 7))
        if (nh + 2 * nkv) * hd * H * es > max_weight_bytes:
            continue
        kvdt = ("f32", "f16")[int(rng.integers(2))]
        n_ctx = int(rng.integers(1, 65))
        pos = int(rng.integers(0, n_ctx))
        cls = CLASSES[int(rng.integers(2))]
        out.append((H, nh, nkv, hd, wdt, kvdt, n_ctx, pos, cls))
    return out


SHAPES = fuzz_shapes()


def shape_id(s):
    return "H%d_h%d_kv%d_d%d_%s_%s_%s" % (s[0], s[1], s[2], s[3], s[4], s[5],
                                          "concat" if s[8] == Q.QKV_CLASS_CONCAT else "mixed")


@pytest.mark.parametrize("shape", SHAPES, ids=shape_id)
def test_random_shape_matches_oracle(orc, qkv, shape):
    H, nh, nkv, hd, wdt, kvdt, n_ctx, pos, cls = shape
    L = HostLayer(H, nh, nkv, hd, wdt, layer=17)
    x = L.x(pos)
    kk0, vv0 = canary(n_ctx, L.nkt, kvdt, 41), canary(n_ctx, L.nkt, kvdt, 42)
    plan = make_plan(L, kvdt, n_ctx, wdt, cls)
    got = run_gpu(L, plan, cls, x, pos, kk0, vv0)
    want = oracle_run(orc, L, x, pos, kk0, vv0)
    assert want[0] == 0
    compare(L, got, want, pos, "random shape %s" % (shape_id(shape),))
    assert Q.qkv_check_device_error()[0] == 0
