"""Seeded random prefill shapes against the per-token CPU oracle.

The hand-picked shapes of test_prefill_gpu.py cover heads of 64 and 128 rows; these add
heads of 192 and 256 rows (three and four pair tiles per head, so a cluster's two pair
tiles can belong to two heads), odd and even pair-tile counts (clusters of 1 and 2 CTAs),
one or two token tiles with ragged last tiles, hidden sizes that leave a ragged last K
block, and both cache types.  The generator is seeded, so every run sees the same shapes.
"""
import numpy as np
import pytest

from qkv_rope_kv_gb300 import synth
from gpu_helpers import canary
from test_prefill_gpu import check, oracle_prefill, run_prefill

pytestmark = pytest.mark.gpu


def fuzz_shapes(n=12, seed=20261203, max_weight_bytes=24 << 20):
    """(nt, H, nh, nkv, hd, n_ctx, kv dtype) tuples."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        hd = 64 * int(rng.integers(1, 5))
        nkv = int(rng.integers(1, 4))
        nh = nkv * int(rng.integers(1, 5))
        H = 8 * int(rng.integers(8, 376))
        if (nh + 2 * nkv) * hd * H * 2 > max_weight_bytes:
            continue
        nt = int(rng.integers(1, 201))
        n_ctx = nt + int(rng.integers(0, 64))
        kvdt = ("f32", "f16")[int(rng.integers(2))]
        out.append((nt, H, nh, nkv, hd, n_ctx, kvdt))
    return out


SHAPES = fuzz_shapes()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "nt%d_H%d_h%d_kv%d_d%d_%s" % (s[:5] + (s[6],)))
def test_random_prefill_matches_oracle(orc, qkv, shape):
    import qkv_rope_kv_gb300 as Q
    nt, H, nh, nkv, hd, n_ctx, kvdt = shape
    R = (nh + 2 * nkv) * hd
    W = synth.weight_rows(0, 21, 0, R, H, "bf16")
    b = synth.bias(0, 21, R)
    X = synth.prefill_x(0, 21, nt, H)
    positions = np.random.default_rng(nt * 7 + H).permutation(n_ctx)[:nt].astype(np.int32)
    kk0, vv0 = canary(n_ctx, nkv * hd, kvdt, 51), canary(n_ctx, nkv * hd, kvdt, 52)
    got = run_prefill(H, nh, nkv, hd, n_ctx, kvdt, X, W, b, positions, kk0, vv0)
    tokens = range(nt) if nt <= 48 else sorted(np.random.default_rng(nt).choice(nt, 48, replace=False))
    want = oracle_prefill(orc, X, W, b, positions, nh, nkv, hd, kk0, vv0, tokens=tokens)
    check(nh, nkv, hd, got, want, positions, "random prefill %s" % (shape,))
    assert Q.qkv_check_device_error()[0] == 0
