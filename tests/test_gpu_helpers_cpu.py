"""The GPU parity rules themselves, on hand-made arrays (no GPU): each accepts what the
stated tolerance allows and rejects a plausible mistake just past it."""
import numpy as np
import pytest

import gpu_helpers as gh


@pytest.fixture(autouse=True)
def _own_records():
    """These hand-made comparisons stay out of the session's parity summary."""
    n = len(gh.RECORDS)
    yield
    del gh.RECORDS[n:]


def test_floored_rule_bounds():
    o = np.array([1.0, -2.0, 0.5, 1e-5, 0.0], np.float64)
    rms = float(np.sqrt(np.mean(o * o)))
    g = o.copy()
    g[1] *= 1 + 0.9e-4                      # 0.9e-4 relative on a large value: inside
    g[3] += 0.9e-4 * gh.RMS_FLOOR * rms     # below the floor: absolute 1e-6 rms
    gh.assert_f32_close(g.astype(np.float32), o.astype(np.float32), "inside")
    g2 = o.copy()
    g2[2] *= 1 + 2e-4                        # 2e-4 relative on a value above the floor
    with pytest.raises(AssertionError):
        gh.assert_f32_close(g2.astype(np.float32), o.astype(np.float32), "relative")
    g3 = o.copy()
    g3[3] += 3e-4 * gh.RMS_FLOOR * rms       # three times the absolute bound below the floor
    with pytest.raises(AssertionError):
        gh.assert_f32_close(g3.astype(np.float32), o.astype(np.float32), "absolute")
    with pytest.raises(AssertionError):
        gh.assert_f32_close(np.array([np.nan], np.float32), np.array([1.0], np.float32), "nan")


def test_f16_spacing_matches_numpy():
    v = np.float16(np.array([1.0, 0.75, 2.0 ** -14, 2.0 ** -20, 60000.0, 3.0e-3], np.float64))
    want = np.abs(np.nextafter(v, np.float16(np.inf)).astype(np.float64) - v.astype(np.float64))
    assert np.array_equal(gh.f16_spacing(v.astype(np.float64)), want)


def test_f16_rule():
    o = np.array([1.0, -0.5, 0.25, 1e-4, -2e-5], np.float64)
    codes = o.astype(np.float16).view(np.uint16)
    up1 = codes.copy()
    up1[0] += 1                               # one ulp: accepted everywhere
    gh.assert_f16_close(up1, codes, o, "one ulp")
    up2 = codes.copy()
    up2[2] += 2                               # two ulps on a value at or above the floor: rejected
    with pytest.raises(AssertionError):
        gh.assert_f16_close(up2, codes, o, "two ulps")
    tiny = codes.copy()
    tiny[4] += 2                              # two ulps (2^-24 each) on a value below the floor
    n0 = len(gh.RECORDS)
    gh.assert_f16_close(tiny, codes, o, "below floor")
    rec = gh.RECORDS[n0]
    assert rec["accepted_via_floor"] == 1 and rec["max_ulp_via_floor"] == 2
    assert rec["max_ulp_at_or_above_floor"] == 0
    far = codes.copy()
    far[4] += 400                             # far beyond the absolute bound
    with pytest.raises(AssertionError):
        gh.assert_f16_close(far, codes, o, "far")


def test_kv_region_untouched_rows_bit_exact():
    want = gh.canary(4, 8, "f16")
    got = want.copy()
    got[2, 3] ^= 1                            # a stray write to a row that must stay untouched
    with pytest.raises(AssertionError):
        gh.assert_kv_region(got, want, 1, "stray")
    n0 = len(gh.RECORDS)
    gh.assert_kv_region(want.copy(), want, None, "untouched")
    assert "(4 rows)" in gh.parity_summary(gh.RECORDS[n0:])


def test_product_rule_floor_from_factors():
    """o = s * u: where u is tiny and s large, the floor comes from |s| rms(u), so an absolute
    error of 0.5e-4 * that passes; twice the bound fails."""
    s = np.array([3.0, 0.5, 1.0, 2.0])
    u = np.array([1e-4, 1.0, -1.0, 0.5])
    o = s * u
    fl = gh.RMS_FLOOR * (np.abs(s) * np.sqrt(np.mean(u * u)) + np.sqrt(np.mean(s * s)) * np.abs(u))
    g = o.copy()
    g[0] += 0.5e-4 * fl[0]
    gh.assert_product_close(g.astype(np.float32), o.astype(np.float32), s, u, "inside")
    g[0] = o[0] + 2e-4 * fl[0]
    with pytest.raises(AssertionError):
        gh.assert_product_close(g.astype(np.float32), o.astype(np.float32), s, u, "outside")
