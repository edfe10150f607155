"""Pins for the CPU oracle: facts fixed by the pages or by mathematics.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with the fact it checks.  ``test_oracle_pins.py``
runs them on the real oracle; ``test_oracle_mutants.py`` runs them on copies
of the oracle with a planted mistake and requires that some pin fails.

None of these re-types the oracle's own formula: they use closed forms
(rotation of unit vectors, hand-derived sums), invariants (norms, relative
position, composition), library routines on special cases (numpy's IEEE f32
multiply and f16 conversion, float64 dot products), arbitrary-precision
evaluation (mpmath) and numbers printed on the pages (tests/golden).
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32_bits(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def bf16_bits_exact(vals) -> np.ndarray:
    """bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(vals, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def read_golden(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- projection

def pin_matvec_closed_form(orc):
    """W[r,c] = r - c, x[c] = c + 1 (4 x 8):
    y[r] = sum_c (r - c)(c + 1) = r * sum(c + 1) - sum(c^2 + c) = 36 r - (140 + 28) = 36 r - 168.
    Small integers are exact in f32 and bf16, so both weight encodings must give it exactly."""
    r = np.arange(4)[:, None]
    c = np.arange(8)[None, :]
    W = (r - c).astype(np.float32)
    x = (np.arange(8) + 1).astype(np.float32)
    expect = np.array([36 * i - 168 for i in range(4)], dtype=np.float64)
    assert np.array_equal(orc.matvec(W, x), expect)
    assert np.array_equal(orc.matvec(bf16_bits_exact(W), x), expect)


def pin_matvec_identity_and_single_entry(orc):
    x = np.array([1.5, -2.0, 0.25, 3.0, -0.125, 8.0, 0.0, -1.0], dtype=np.float32)
    assert np.array_equal(orc.matvec(np.eye(8, dtype=np.float32), x), x.astype(np.float64))
    # one non-zero at (row 1, column 6) of a 4 x 8 matrix: only y[1] = 2 * x[6] ... with x[6]
    # replaced to be non-zero; a transposed read would put it elsewhere.
    x2 = x.copy()
    x2[6] = 0.75
    W = np.zeros((4, 8), dtype=np.float32)
    W[1, 6] = 2.0
    y = orc.matvec(W, x2)
    assert np.array_equal(y, np.array([0.0, 1.5, 0.0, 0.0]))


def pin_matvec_vs_float64_dot(orc):
    """Random shapes against numpy's float64 dot product (a library routine)."""
    rng = np.random.default_rng(1)
    for R, H in ((37, 53), (3, 1000), (64, 7)):
        W = rng.standard_normal((R, H)).astype(np.float32)
        x = rng.standard_normal(H).astype(np.float32)
        ref = W.astype(np.float64) @ x.astype(np.float64)
        y = orc.matvec(W, x)
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
        Wb = (W.view(np.uint32) >> 16).astype(np.uint16)        # truncate to bf16
        Wb_val = (Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.allclose(orc.matvec(Wb, x), Wb_val @ x.astype(np.float64), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- frequencies

def _mp_round_f32(v):
    """Correctly rounded f32 of an mpmath number (nearest, ties to even)."""
    import mpmath
    f = np.float32(float(v))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        err = abs(mpmath.mpf(float(cand)) - v)
        key = (err, int(np.asarray(cand, np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def pin_inv_freq_correctly_rounded(orc):
    import mpmath
    mpmath.mp.dps = 60
    for hd in (4, 64, 128):
        for base in (1.0e4, 1.0e6):
            for fs in (1.0, 0.25):
                tab = orc.inv_freq_table(hd, base, fs)
                for d in range(hd // 2):
                    exact = mpmath.mpf(fs) * mpmath.power(mpmath.mpf(base), mpmath.mpf(-2 * d) / hd)
                    assert f32_bits(tab[d]) == f32_bits(_mp_round_f32(exact)), (hd, base, fs, d)
    # closed forms: d = 0 gives freq_scale; 10000^(-2/4) = 1/100
    assert orc.inv_freq(0, 128, 1.0e6, 1.0) == np.float32(1.0)
    assert f32_bits(orc.inv_freq(1, 4, 1.0e4, 1.0)) == f32_bits(np.float32(0.01))


def pin_theta_is_f32_product(orc):
    """The angle is the IEEE single-precision product pos * inv_freq."""
    rng = np.random.default_rng(2)
    for _ in range(2000):
        pos = int(rng.integers(0, 1 << 20))
        f = np.float32(rng.uniform(1e-7, 1.0))
        assert f32_bits(orc.theta(pos, f)) == f32_bits(np.float32(pos) * f)
    for pos in (0, 1, 17, 1641, 3254, 4095):
        assert orc.theta(pos, np.float32(1.0)) == np.float32(pos)


# ---------------------------------------------------------------- rotation

def pin_rope_identity_at_pos0(orc):
    rng = np.random.default_rng(3)
    for _ in range(500):
        y0, y1 = rng.standard_normal(2) * 3
        b0, b1 = rng.standard_normal(2).astype(np.float32)
        f = np.float32(rng.uniform(1e-6, 1.0))
        r0, r1 = orc.rope_pair(y0, y1, b0, b1, 0, f)
        assert f32_bits(r0) == f32_bits(np.float32(y0 + float(b0)))
        assert f32_bits(r1) == f32_bits(np.float32(y1 + float(b1)))


def pin_rope_unit_vectors(orc):
    """With frequency 1 the angle is pos radians exactly; (1,0) maps to (cos, sin) and (0,1) to
    (-sin, cos): the counter-clockwise rotation of the neox pairing."""
    for pos in (1, 2, 3, 17, 100, 1641, 3254):
        c, s = math.cos(float(pos)), math.sin(float(pos))
        r0, r1 = orc.rope_pair(1.0, 0.0, 0.0, 0.0, pos, 1.0)
        assert abs(float(r0) - c) < 1e-7 and abs(float(r1) - s) < 1e-7, pos
        r0, r1 = orc.rope_pair(0.0, 1.0, 0.0, 0.0, pos, 1.0)
        assert abs(float(r0) + s) < 1e-7 and abs(float(r1) - c) < 1e-7, pos


def pin_rope_preserves_pair_norm(orc):
    rng = np.random.default_rng(4)
    for _ in range(2000):
        y0, y1 = rng.standard_normal(2)
        b0, b1 = (rng.standard_normal(2) * 0.1).astype(np.float32)
        pos = int(rng.integers(0, 5000))
        f = orc.inv_freq(int(rng.integers(0, 64)), 128, 1.0e6)
        r0, r1 = orc.rope_pair(y0, y1, b0, b1, pos, f)
        n_in = (y0 + float(b0)) ** 2 + (y1 + float(b1)) ** 2
        n_out = float(r0) ** 2 + float(r1) ** 2
        assert abs(n_out - n_in) <= 1e-6 * n_in + 1e-12


def pin_rope_composition(orc):
    """rope(rope(x, a), b) == rope(x, a + b) when the angle is exact (frequency 1)."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        x0, x1 = rng.standard_normal(2)
        a, b = (int(v) for v in rng.integers(0, 200, size=2))
        t0, t1 = orc.rope_pair(x0, x1, 0.0, 0.0, a, 1.0)
        u0, u1 = orc.rope_pair(float(t0), float(t1), 0.0, 0.0, b, 1.0)
        w0, w1 = orc.rope_pair(x0, x1, 0.0, 0.0, a + b, 1.0)
        scale = math.hypot(x0, x1)
        assert abs(float(u0) - float(w0)) < 1e-6 * scale and abs(float(u1) - float(w1)) < 1e-6 * scale


def _head_token(orc, yq, yk, pos, hd, base=1.0e4):
    """Run one head of q and one head of k through the token epilogue (bias 0)."""
    y = np.concatenate([yq, yk, np.zeros(hd)])
    kv = np.zeros((pos + 1, hd), np.float32)
    st, q, k, v = orc.token(y, np.zeros(3 * hd, np.float32), 1, 1, hd, base, 1.0, pos, kv, kv.copy())
    assert st == 0
    return q, k


def pin_rope_relative_position(orc):
    """<rope(q, m), rope(k, n)> depends only on m - n."""
    rng = np.random.default_rng(6)
    hd = 64
    for _ in range(40):
        yq, yk = rng.standard_normal(hd), rng.standard_normal(hd)
        m, n = (int(v) for v in rng.integers(0, 32, size=2))
        s = int(rng.integers(1, 32))
        q1, k1 = _head_token(orc, yq, yk, m, hd)
        q1b, k1b = _head_token(orc, yq, yk, n, hd)
        q2, _ = _head_token(orc, yq, yk, m + s, hd)
        _, k2 = _head_token(orc, yq, yk, n + s, hd)
        dot1 = float(np.dot(q1.astype(np.float64), k1b.astype(np.float64)))
        dot2 = float(np.dot(q2.astype(np.float64), k2.astype(np.float64)))
        scale = float(np.linalg.norm(yq) * np.linalg.norm(yk))
        assert abs(dot1 - dot2) < 1e-4 * scale, (m, n, s)


def pin_neox_pairing(orc):
    """A lone 1 at element d of a head rotates into elements d and d + hd/2 only, as
    (cos, sin) of that pair's angle; a lone 1 at d + hd/2 gives (-sin, cos)."""
    nh, nkv, hd, pos, base = 2, 1, 8, 5, 1.0e4
    nqt, nkt = nh * hd, nkv * hd
    R = nqt + 2 * nkt
    for sec_off, n_in_sec in ((0, nqt), (nqt, nkt)):
        for j in range(n_in_sec):
            h, d = divmod(j, hd)
            half = hd // 2
            y = np.zeros(R)
            y[sec_off + j] = 1.0
            kv = np.zeros((8, nkt), np.float32)
            st, q, k, v = orc.token(y, np.zeros(R, np.float32), nh, nkv, hd, base, 1.0, pos, kv,
                                    kv.copy())
            out = q if sec_off == 0 else k
            dd = d % half
            th = float(orc.theta(pos, orc.inv_freq(dd, hd, base)))
            c, s = math.cos(th), math.sin(th)
            lo, hi = h * hd + dd, h * hd + dd + half
            expect = np.zeros(n_in_sec)
            if d < half:
                expect[lo], expect[hi] = c, s
            else:
                expect[lo], expect[hi] = -s, c
            assert np.allclose(out.astype(np.float64), expect, atol=1e-7), (sec_off, j)


# ---------------------------------------------------------------- sections, bias, cache

def pin_sections_and_bias(orc):
    """Concat output rows are q | k | v with k at nqt and v at nqt + nkt (nh != nkv so a v base
    of 2*nkt would be caught).  At pos 0 the outputs are the biased projections; with y = 0 they
    are the bias itself."""
    nh, nkv, hd = 3, 1, 4
    nqt, nkt = nh * hd, nkv * hd
    R = nqt + 2 * nkt
    y = np.arange(R, dtype=np.float64) + 1.0
    kv = np.zeros((2, nkt), np.float32)
    st, q, k, v = orc.token(y, np.zeros(R, np.float32), nh, nkv, hd, 1.0e4, 1.0, 0, kv, kv.copy())
    assert np.array_equal(q, y[:nqt].astype(np.float32))
    assert np.array_equal(k, y[nqt:nqt + nkt].astype(np.float32))
    assert np.array_equal(v, y[nqt + nkt:].astype(np.float32))
    b = (np.arange(R, dtype=np.float32) - 7.0) * 0.5
    st, q, k, v = orc.token(np.zeros(R), b, nh, nkv, hd, 1.0e4, 1.0, 0, kv, kv.copy())
    assert np.array_equal(np.concatenate([q, k, v]), b)
    # a non-zero angle still carries v through untouched by the rotation: v = y_v + b_v
    st, q, k, v = orc.token(y, b, nh, nkv, hd, 1.0e4, 1.0, 1, kv, kv.copy())
    assert np.array_equal(v, (y[nqt + nkt:] + b[nqt + nkt:].astype(np.float64)).astype(np.float32))


def _canary_f32(shape):
    n = int(np.prod(shape))
    return (np.uint32(0x7F800001) + np.arange(n, dtype=np.uint32) % np.uint32(0x3FFFFF)).reshape(
        shape).view(np.float32)


def _canary_f16(shape):
    n = int(np.prod(shape))
    return (np.uint16(0x7C01) + (np.arange(n) % 0x1FF).astype(np.uint16)).reshape(shape)


def pin_kv_layout(orc):
    """Element (pos, j) of a layer's region sits at flat index pos * nkt + j; every other slot
    keeps its bits (a NaN-payload canary per slot)."""
    nh, nkv, hd, n_ctx, pos = 2, 2, 4, 5, 3
    nqt, nkt = nh * hd, nkv * hd
    R = nqt + 2 * nkt
    rng = np.random.default_rng(7)
    y = rng.standard_normal(R)
    b = rng.standard_normal(R).astype(np.float32)
    for f16 in (False, True):
        kk = _canary_f16((n_ctx, nkt)) if f16 else _canary_f32((n_ctx, nkt))
        vv = kk.copy()[::-1].copy()
        k0, v0 = kk.copy(), vv.copy()
        st, q, k, v = orc.token(y, b, nh, nkv, hd, 1.0e4, 1.0, pos, kk, vv)
        assert st == 0
        flat_k, flat_v = kk.reshape(-1), vv.reshape(-1)
        for i in range(n_ctx * nkt):
            p, j = divmod(i, nkt)
            if p == pos:
                want_k = orc.f32_to_f16(k[j]) if f16 else f32_bits(k[j])
                want_v = orc.f32_to_f16(v[j]) if f16 else f32_bits(v[j])
                got_k = int(flat_k[i]) if f16 else f32_bits(flat_k[i])
                got_v = int(flat_v[i]) if f16 else f32_bits(flat_v[i])
                assert got_k == want_k and got_v == want_v, i
            else:
                a, c = (flat_k[i], k0.reshape(-1)[i]) if f16 else (f32_bits(flat_k[i]), f32_bits(k0.reshape(-1)[i]))
                assert a == c, i
                a, c = (flat_v[i], v0.reshape(-1)[i]) if f16 else (f32_bits(flat_v[i]), f32_bits(v0.reshape(-1)[i]))
                assert a == c, i


def pin_pos_out_of_range(orc):
    """A position outside [0, n_ctx) is an error: nothing is stored, status is reported."""
    nh, nkv, hd, n_ctx = 1, 1, 4, 3
    R = (nh + 2 * nkv) * hd
    y = np.arange(R, dtype=np.float64)
    for pos in (-1, n_ctx, n_ctx + 10):
        kk = _canary_f32((n_ctx, nkv * hd))
        vv = kk.copy()
        k0 = kk.copy()
        st, q, k, v = orc.token(y, np.zeros(R, np.float32), nh, nkv, hd, 1.0e4, 1.0, pos, kk, vv)
        assert st == 1
        assert np.array_equal(f32_bits(kk), f32_bits(k0)) and np.array_equal(f32_bits(vv), f32_bits(k0))
    kk = np.zeros((n_ctx, nkv * hd), np.float32)
    st, *_ = orc.token(y, np.zeros(R, np.float32), nh, nkv, hd, 1.0e4, 1.0, n_ctx - 1, kk, kk.copy())
    assert st == 0


# ---------------------------------------------------------------- f16 conversion

F16_HAND = [
    # (f32 value, f16 code, derivation from the binary16 definition)
    (1.0, 0x3C00, "exponent 15, fraction 0"),
    (1.0 + 2.0 ** -10, 0x3C01, "one ulp above 1"),
    (1.0 + 2.0 ** -11, 0x3C00, "tie between 1 and 1+2^-10: even fraction 0"),
    (1.0 + 3 * 2.0 ** -11, 0x3C02, "tie between fraction 1 and 2: even 2"),
    (1.0 + 2.0 ** -11 + 2.0 ** -20, 0x3C01, "just above the tie rounds up"),
    (-2.0, 0xC000, "sign bit, exponent 16"),
    (65504.0, 0x7BFF, "largest finite"),
    (65519.0, 0x7BFF, "below the 65520 midpoint"),
    (65520.0, 0x7C00, "midpoint to 65536, which is not representable: infinity"),
    (2.0 ** -14, 0x0400, "smallest normal"),
    (2.0 ** -24, 0x0001, "smallest subnormal"),
    (2.0 ** -25, 0x0000, "tie between 0 and 2^-24: even 0"),
    (3 * 2.0 ** -26, 0x0001, "0.75 of the smallest subnormal rounds up"),
    (3 * 2.0 ** -25, 0x0002, "tie between 1 and 2 subnormal quanta: even 2"),
    (-0.0, 0x8000, "negative zero keeps its sign"),
    (float("inf"), 0x7C00, "infinity"),
    (float("-inf"), 0xFC00, "negative infinity"),
]


def pin_f16_hand_cases(orc):
    for val, code, why in F16_HAND:
        assert orc.f32_to_f16(val) == code, (val, hex(code), why)
    nan = orc.f32_to_f16(float("nan"))
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x03FF) != 0


def pin_f16_vs_numpy(orc):
    """numpy's float32 -> float16 cast rounds to nearest even: compare on random values over the
    whole f16 range and on every exact midpoint between adjacent f16 values."""
    rng = np.random.default_rng(8)
    vals = (rng.standard_normal(4000) * np.exp2(rng.integers(-28, 17, 4000))).astype(np.float32)
    codes = np.arange(0, 0x7C00, 7, dtype=np.uint32)
    lo = codes.astype(np.uint16).view(np.float16).astype(np.float64)
    hi = (codes + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (lo + hi) / 2)  # midpoints exact in f32
    with np.errstate(over="ignore"):
        ref = np.concatenate([vals, mids, -mids]).astype(np.float16).view(np.uint16)
    for v, r in zip(np.concatenate([vals, mids, -mids]), ref):
        assert orc.f32_to_f16(v) == int(r), v


# ---------------------------------------------------------------- class and token equivalences

def pin_mixed_equals_concat(orc):
    rng = np.random.default_rng(9)
    nh, nkv, hd, H = 4, 2, 8, 40
    nqt, nkt = nh * hd, nkv * hd
    W = rng.standard_normal((nqt + 2 * nkt, H)).astype(np.float32) * 0.1
    x = rng.standard_normal(H).astype(np.float32)
    b = rng.standard_normal(nqt + 2 * nkt).astype(np.float32) * 0.1
    ka, va = np.zeros((9, nkt), np.float32), np.zeros((9, nkt), np.float32)
    kb, vb = ka.copy(), va.copy()
    r1 = orc.decode(W, x, b, nh, nkv, hd, 1.0e6, 1.0, 6, ka, va)
    r2 = orc.decode_mixed(W[:nqt], W[nqt:nqt + nkt], W[nqt + nkt:], x, b, nh, nkv, hd, 1.0e6, 1.0,
                          6, kb, vb)
    for a, c in zip(r1[1:], r2[1:]):
        assert np.array_equal(f32_bits(a), f32_bits(c))
    assert np.array_equal(f32_bits(ka), f32_bits(kb)) and np.array_equal(f32_bits(va), f32_bits(vb))


def pin_prefill_equals_decode(orc):
    rng = np.random.default_rng(10)
    nh, nkv, hd, H, nt = 2, 1, 8, 24, 5
    nqt, nkt = nh * hd, nkv * hd
    R = nqt + 2 * nkt
    W = bf16_bits_exact(np.round(rng.standard_normal((R, H)) * 64) / 256)
    X = bf16_bits_exact(np.round(rng.standard_normal((nt, H)) * 32) / 16)
    b = rng.standard_normal(R).astype(np.float32) * 0.1
    positions = np.array([0, 3, 4, 7, 9], np.int32)
    kp, vp = np.zeros((10, nkt), np.uint16), np.zeros((10, nkt), np.uint16)
    st, Y = orc.prefill(X, W, b, positions, nh, nkv, hd, 1.0e4, 1.0, kp, vp)
    assert st == 0
    kd, vd = np.zeros_like(kp), np.zeros_like(vp)
    for t in range(nt):
        x = (X[t].astype(np.uint32) << 16).view(np.float32)
        st, q, k, v = orc.decode(W, x, b, nh, nkv, hd, 1.0e4, 1.0, int(positions[t]), kd, vd)
        assert np.array_equal(f32_bits(Y[t]), f32_bits(np.concatenate([q, k, v])))
    assert np.array_equal(kp, kd) and np.array_equal(vp, vd)


# ---------------------------------------------------------------- FusedFFN

def pin_silu_special_values(orc):
    """SiLU(v) = v * sigmoid(v): SiLU(0) = 0; sigmoid(ln 3) = 3/4, so SiLU(ln 3) = 0.75 ln 3;
    SiLU(v) - SiLU(-v) = v (since sigmoid(v) + sigmoid(-v) = 1); SiLU(v) -> v for large v
    and -> v e^v for very negative v; other points against mpmath."""
    import mpmath
    mpmath.mp.dps = 50
    assert orc.silu(0.0) == 0.0
    ln3 = math.log(3.0)
    assert abs(orc.silu(ln3) - 0.75 * ln3) <= 1e-15 * ln3
    for v in (0.125, 1.0, 2.5, 7.0, 19.0):
        assert abs((orc.silu(v) - orc.silu(-v)) - v) <= 1e-14 * v, v
    assert abs(orc.silu(40.0) - 40.0) <= 1e-13
    assert abs(orc.silu(-40.0) - (-40.0 * math.exp(-40.0))) <= 1e-12 * 40.0 * math.exp(-40.0)
    for v in (-3.75, -0.5, 0.3, 1.7, 6.25):
        exact = mpmath.mpf(v) / (1 + mpmath.exp(-mpmath.mpf(v)))
        assert abs(orc.silu(v) - float(exact)) <= 1e-15 * max(1.0, abs(float(exact))), v


def _ffn_hand_case():
    """nf = 3, H = 4, small integers and halves: exact in f32, bf16 and float64.
    gate_i = sum_c (i - c) x_c and up_i = sum_c (i + 2c + 1) x_c are all distinct."""
    nf, H = 3, 4
    i = np.arange(nf)[:, None]
    c = np.arange(H)[None, :]
    Wg = (i - c).astype(np.float32)
    Wu = (i + 2 * c + 1).astype(np.float32)
    x = np.array([1.0, -1.0, 2.0, 0.5], dtype=np.float32)
    g = Wg.astype(np.float64) @ x.astype(np.float64)
    u = Wu.astype(np.float64) @ x.astype(np.float64)
    assert len(set(g.tolist()) | set(u.tolist())) == 2 * nf
    return np.concatenate([Wg, Wu]), x, g, u


def pin_ffn_gate_up_pairing(orc):
    """out[i] = SiLU(gate_i) * up_i with gate from row i and up from row nf + i of the concat
    weight: checked against mpmath at correctly rounded f32, for f32 and bf16 weights."""
    import mpmath
    mpmath.mp.dps = 50
    W, x, g, u = _ffn_hand_case()
    want = np.array([_mp_round_f32(mpmath.mpf(gi) / (1 + mpmath.exp(-mpmath.mpf(gi))) * mpmath.mpf(ui))
                     for gi, ui in zip(g, u)], dtype=np.float32)
    for enc in (W, bf16_bits_exact(W)):
        got = orc.ffn_swiglu(enc, x)
        assert got.shape == (3,)
        # the double-precision result may sit one f32 ulp from the exact one only at a tie
        assert np.all(np.abs(f32_bits(got).astype(np.int64) - f32_bits(want).astype(np.int64)) <= 1), (got, want)


def pin_ffn_zero_gate_and_unit_up(orc):
    """A zero gate row gives 0 whatever the up row; a gate row of e_0 with x_0 = ln 3 and an
    up row of 4 e_0 gives SiLU(ln 3) * 4 ln 3 = 3 (ln 3)^2."""
    ln3 = np.float32(math.log(3.0))
    x = np.array([ln3, 5.0], dtype=np.float32)
    W = np.array([[0.0, 0.0],    # gate 0: zero
                  [1.0, 0.0],    # gate 1: x0
                  [7.0, -3.0],   # up 0: anything
                  [4.0, 0.0]],   # up 1: 4 x0
                 dtype=np.float32)
    out = orc.ffn_swiglu(W, x)
    assert out[0] == 0.0
    want = 3.0 * float(ln3) ** 2
    assert abs(float(out[1]) - want) <= 2e-7 * want


# ---------------------------------------------------------------- RMSNorm prologue

def pin_rmsnorm_closed_forms(orc):
    """h = 3 * ones, w = ones, eps = 0: mean(h^2) = 9, so x = 1 exactly; h = ones, eps = 3:
    x = 1 / sqrt(1 + 3) = 0.5 exactly; h = 0: x = 0 for any eps > 0; h = [3, 4]: against mpmath."""
    import mpmath
    mpmath.mp.dps = 40
    ones = np.ones(7, np.float32)
    assert np.array_equal(orc.rmsnorm(3 * ones, ones, 0.0), ones)
    assert np.array_equal(orc.rmsnorm(-3 * ones, ones, 0.0), -ones)
    assert np.array_equal(orc.rmsnorm(ones, ones, 3.0), 0.5 * ones)
    assert np.array_equal(orc.rmsnorm(np.zeros(5, np.float32), np.ones(5, np.float32), 1e-6), np.zeros(5, np.float32))
    h = np.array([3.0, 4.0], np.float32)
    want = [_mp_round_f32(mpmath.mpf(v) / mpmath.sqrt(mpmath.mpf(25) / 2 + mpmath.mpf("1e-6"))) for v in (3, 4)]
    got = orc.rmsnorm(h, np.ones(2, np.float32), 1e-6)
    assert np.all(np.abs(f32_bits(got).astype(np.int64) - f32_bits(np.array(want, np.float32)).astype(np.int64)) <= 1)


def pin_rmsnorm_scale_and_weight(orc):
    """With eps = 0, scaling h by a power of two leaves x unchanged bit for bit (every sum,
    square and root scales exactly); the weight multiplies element by element."""
    rng = np.random.default_rng(5)
    h = rng.standard_normal(64).astype(np.float32)
    w = np.ones(64, np.float32)
    base = orc.rmsnorm(h, w, 0.0)
    for k in (-3, 1, 5):
        assert np.array_equal(orc.rmsnorm((h * np.float32(2.0 ** k)).astype(np.float32), w, 0.0), base)
    w2 = np.arange(1, 65, dtype=np.float32) / np.float32(8)  # exact in f32
    got = orc.rmsnorm(h, w2, 0.0).astype(np.float64)
    assert np.allclose(got, base.astype(np.float64) * w2, rtol=2e-7, atol=0)
    # the mean is over H: the norm of the normalised vector is sqrt(H)
    assert abs(float(np.sqrt(np.sum(base.astype(np.float64) ** 2))) - 8.0) <= 1e-5


def _qkn(orc, yq, yk, yv, bias, wq, wk, eps, pos, hd, n_ctx=4, base=1.0e4):
    """token_qknorm on hand-made sections (f32 cache of n_ctx rows)."""
    nh, nkv = len(yq) // hd, len(yk) // hd
    y = np.concatenate([yq, yk, yv]).astype(np.float64)
    kk = np.zeros((n_ctx, nkv * hd), np.float32)
    vv = np.zeros((n_ctx, nkv * hd), np.float32)
    st, q, k, v = orc.token_qknorm(y, np.asarray(bias, np.float32), np.asarray(wq, np.float32),
                                   np.asarray(wk, np.float32), eps, nh, nkv, hd, base, 1.0, pos, kk, vv)
    return st, q, k, v, kk, vv


def pin_qknorm_closed_forms(orc):
    """FusedQkvNorm with hd = 2 at pos 0 (no rotation): a head z = (1, 1) has RMS 1, so q = w
    exactly; z = (0.5, 0.5) gives k = w_k; the bias is added before the norm (y = 0 with
    bias (2, 2) still normalises to w); eps = 3 on z = (1, 1) gives 1 / sqrt(1 + 3) = 0.5;
    two q heads are normalised separately; v is y + b, untouched by the norm."""
    wq, wk = [1.0, 2.0], [3.0, 0.25]
    st, q, k, v, kk, vv = _qkn(orc, [1, 1], [0.5, 0.5], [3, 4], [0, 0, 0, 0, 0.5, -1], wq, wk, 0.0, 0, 2)
    assert st == 0
    assert np.array_equal(q, np.float32(wq)) and np.array_equal(k, np.float32(wk))
    assert np.array_equal(v, np.float32([3.5, 3.0]))
    assert np.array_equal(kk[0], k) and np.array_equal(vv[0], v) and not kk[1:].any()
    st, q, k, v, _, _ = _qkn(orc, [0, 0], [0, 0], [0, 0], [2, 2, -4, -4, 0, 0], wq, wk, 0.0, 0, 2)
    assert np.array_equal(q, np.float32(wq)) and np.array_equal(k, -np.float32(wk))
    st, q, k, v, _, _ = _qkn(orc, [1, 1], [1, 1], [0, 0], np.zeros(6), wq, wk, 3.0, 0, 2)
    assert np.array_equal(q, np.float32([0.5, 1.0])) and np.array_equal(k, np.float32([1.5, 0.125]))
    # head 0 = (3, 4) (RMS sqrt(12.5)), head 1 = (1, 1): head 1 is w whatever head 0 holds
    st, q, k, v, _, _ = _qkn(orc, [3, 4, 1, 1], [1, 1], [0, 0], np.zeros(8), wq, wk, 0.0, 0, 2)
    assert np.array_equal(q[2:], np.float32(wq))
    want0 = np.float32(np.array([3.0, 8.0]) / np.sqrt(12.5))
    assert np.all(np.abs(f32_bits(q[:2]).astype(np.int64) - f32_bits(want0).astype(np.int64)) <= 1)


def pin_qknorm_norm_before_rotation(orc):
    """The norm and its weight act before the rotation: z = (1, 1), w = (1, 2), eps = 0 at
    pos 7 gives n = (1, 2) rotated by theta, i.e. (cos - 2 sin, sin + 2 cos), not the
    weighted rotation of (1, 1)."""
    hd, pos, base = 2, 7, 1.0e4
    th = float(orc.theta(pos, orc.inv_freq(0, hd, base)))
    c, s_ = np.cos(th), np.sin(th)
    st, q, _, _, _, _ = _qkn(orc, [1, 1], [1, 1], [0, 0], np.zeros(6), [1, 2], [1, 1], 0.0, pos, hd)
    want = np.float32([c - 2 * s_, s_ + 2 * c])
    assert np.array_equal(q, want)
    other = np.float32([c - s_, 2 * (s_ + c)])
    assert not np.allclose(q, other, rtol=1e-3)


def pin_qknorm_invariants(orc):
    """Random heads (hd = 8, 3 q heads, 2 k heads), eps = 0: scaling the projection by a power
    of two changes no bit of q or k; with w = 1 every rotated head has sum of squares hd; a
    head of +-1 entries has RMS exactly 1, so with w = 1 the stage equals the plain stage
    (token) bit for bit; an out-of-range position stores nothing."""
    rng = np.random.default_rng(11)
    hd, nh, nkv, pos = 8, 3, 2, 5
    yq = rng.standard_normal(nh * hd)
    yk = rng.standard_normal(nkv * hd)
    yv = rng.standard_normal(nkv * hd)
    w1 = np.ones(hd)
    wq = rng.uniform(0.5, 1.5, hd)
    bias = np.zeros((nh + 2 * nkv) * hd)
    st, q0, k0, v0, _, _ = _qkn(orc, yq, yk, yv, bias, wq, wq[::-1], 0.0, pos, hd, n_ctx=8)
    for e in (-4, 3):
        f = 2.0 ** e
        _, q1, k1, _, _, _ = _qkn(orc, yq * f, yk * f, yv, bias, wq, wq[::-1], 0.0, pos, hd, n_ctx=8)
        assert np.array_equal(q1, q0) and np.array_equal(k1, k0)
    _, q2, k2, _, _, _ = _qkn(orc, yq, yk, yv, bias, w1, w1, 0.0, pos, hd, n_ctx=8)
    for h in range(nh):
        assert abs(float(np.sum(q2[h * hd:(h + 1) * hd].astype(np.float64) ** 2)) - hd) <= 1e-5
    sq = np.where(rng.standard_normal(nh * hd) > 0, 1.0, -1.0)
    sk = np.where(rng.standard_normal(nkv * hd) > 0, 1.0, -1.0)
    b = rng.standard_normal((nh + 2 * nkv) * hd).astype(np.float32)
    b[: (nh + nkv) * hd] = 0
    st, q3, k3, v3, kk3, vv3 = _qkn(orc, sq, sk, yv, b, w1, w1, 0.0, pos, hd, n_ctx=8)
    kk = np.zeros((8, nkv * hd), np.float32)
    vv = np.zeros((8, nkv * hd), np.float32)
    st2, qt, kt, vt = orc.token(np.concatenate([sq, sk, yv]), b, nh, nkv, hd, 1.0e4, 1.0, pos, kk, vv)
    assert st == st2 == 0
    assert np.array_equal(q3, qt) and np.array_equal(k3, kt) and np.array_equal(v3, vt)
    assert np.array_equal(kk3, kk) and np.array_equal(vv3, vv)
    st, _, _, _, kk4, vv4 = _qkn(orc, yq, yk, yv, bias, wq, wq, 0.0, 8, hd, n_ctx=8)
    assert st == 1 and not kk4.any() and not vv4.any()


def _qkn_decode_case(orc, w_dtype, pos):
    """The concat FusedQkvNorm stage (projection + norm + rotation + stores) on a hand case,
    H = 3, hd = 2, two q heads, one kv head, integer weights and x = (1, 2, 3), so that the
    projection is exact: q heads (1, 1) and (-2, 2), k head (3, -3), v (5, 7)."""
    W = np.array([[1, 0, 0], [1, 0, 0],       # q head 0: (1, 1), RMS 1
                  [0, -1, 0], [0, 1, 0],      # q head 1: (-2, 2), RMS 2
                  [0, 0, 1], [0, 0, -1],      # k head:   (3, -3), RMS 3
                  [1, 2, 0], [1, 0, 2]],      # v:        (5, 7)
                 np.float32)
    if w_dtype == "bf16":
        W = bf16_bits_exact(W)
    x = np.array([1, 2, 3], np.float32)
    bias = np.array([0, 0, 0, 0, 0, 0, 0.5, -1], np.float32)
    wq, wk = np.float32([1.0, 2.0]), np.float32([3.0, 0.25])
    kk = np.zeros((4, 2), np.float32)
    vv = np.zeros((4, 2), np.float32)
    st, q, k, v = orc.decode_qknorm(W, x, bias, wq, wk, 0.0, 2, 1, 2, 1.0e4, 1.0, pos, kk, vv)
    return st, q, k, v, kk, vv


def pin_qknorm_decode_hand_case(orc):
    """The concat wrapper of FusedQkvNorm, through the projection: each head normalises to
    (+-1, +-1), so at pos 0 q = (w_q, -w_q[0], w_q[1]), k = (w_k[0], -w_k[1]) and v = y + b =
    (5.5, 6), with k and v stored in row 0 only (f32 and bf16 weights).  At pos 2 the pair
    angle is exactly 2 rad (pair index 0 has frequency freq_scale = 1): each normalised pair
    (n0, n1) becomes (n0 cos 2 - n1 sin 2, n0 sin 2 + n1 cos 2), stored in row 2."""
    wq, wk = np.float32([1.0, 2.0]), np.float32([3.0, 0.25])
    for w_dtype in ("f32", "bf16"):
        st, q, k, v, kk, vv = _qkn_decode_case(orc, w_dtype, 0)
        assert st == 0
        assert np.array_equal(q, np.float32([wq[0], wq[1], -wq[0], wq[1]]))
        assert np.array_equal(k, np.float32([wk[0], -wk[1]]))
        assert np.array_equal(v, np.float32([5.5, 6.0]))
        assert np.array_equal(kk[0], k) and np.array_equal(vv[0], v) and not kk[1:].any() and not vv[1:].any()
    c, s_ = np.cos(2.0), np.sin(2.0)

    def rot(n0, n1):
        return np.float32([n0 * c - n1 * s_, n0 * s_ + n1 * c])

    st, q, k, v, kk, vv = _qkn_decode_case(orc, "f32", 2)
    assert st == 0
    want_q = np.concatenate([rot(1.0, 2.0), rot(-1.0, 2.0)])
    want_k = rot(3.0, -0.25)
    for got, want in ((q, want_q), (k, want_k)):
        assert np.all(np.abs(f32_bits(got).astype(np.int64) - f32_bits(want).astype(np.int64)) <= 1)
    assert np.array_equal(v, np.float32([5.5, 6.0]))
    assert np.array_equal(kk[2], k) and np.array_equal(vv[2], v)
    assert not kk[[0, 1, 3]].any() and not vv[[0, 1, 3]].any()


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
