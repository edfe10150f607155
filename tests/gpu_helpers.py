"""Helpers for the GPU parity tests: seeded layers, device transfer, comparison rules.

Comparison rules (the tolerance the stage's arithmetic supports):
  * cache addressing and untouched slots: bit-exact;
  * q / k / v and f32 cache values, per section: |g - o| <= 1e-4 * max(|o|, 1e-2 * rms(o)),
    i.e. 1e-4 relative for every value at or above one hundredth of the section's RMS
    and 1e-6 * RMS absolute below it, where an f32 accumulation of H products cannot
    keep an elementwise relative bound (its absolute error is ~1e-7 * sqrt(H) * |w| |x|);
  * a product of two such values (the FusedFFN output silu(g) * u): the same bound with
    the floor of element i taken from the factors, 1e-2 * (|s_i| rms(u) + rms(s) |u_i|);
  * f16 cache values: the f16 code within 1 ulp of the oracle's code wherever the
    oracle's f32 value is at or above the output's floor (1e-2 * rms, the prefill's 1e-1);
    below it, within the f32 rule's absolute bound plus one f16 spacing (rounding g and o
    to f16 can add one).
Every comparison is recorded (floored error, unfloored elementwise error, f16 codes
accepted only below the floor and their largest ulp distance), and the session prints
the maxima at its end.
"""
from __future__ import annotations

import json
import os

import numpy as np

from qkv_rope_kv_gb300 import synth

REL_TOL = 1e-4
RMS_FLOOR = 1e-2   # values below RMS_FLOOR * rms(section) are held to an absolute bound
# The prefill's sums run on the tensor cores (tcgen05 kind::f16, f32 accumulation), whose
# additions inside an MMA are not each rounded to nearest as the CUDA-core FMA chains are;
# their error near zero is several times larger (3.5e-6 * rms measured on the 14B shape),
# so prefill outputs take a floor of 1e-1 * rms (an absolute bound of 1e-5 * rms).
PREFILL_RMS_FLOOR = 1e-1

# Every comparison made in this process: dicts with kind, what, and the measured errors.
RECORDS: list = []


def _record(**kw):
    RECORDS.append(kw)
    path = os.environ.get("QKV_PARITY_LOG")
    if path:
        with open(path, "a") as fh:
            fh.write(json.dumps(kw) + "\n")


# ---------------------------------------------------------------- comparison

def _rms(o: np.ndarray) -> float:
    return float(np.sqrt(np.mean(o * o))) if o.size else 0.0


def floored_rel_err(got, want, floor: float = RMS_FLOOR) -> float:
    """max |g - o| / max(|o|, floor * rms(o)) over the section."""
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    if o.size == 0:
        return 0.0
    den = np.maximum(np.abs(o), max(floor * _rms(o), 1e-30))
    return float(np.max(np.abs(g - o) / den))


def elementwise_rel_err(got, want) -> float:
    """Unfloored max |g-o|/|o| over |o| > 0 (recorded, not gated)."""
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    m = o != 0
    return float(np.max(np.abs(g[m] - o[m]) / np.abs(o[m]))) if m.any() else 0.0


def assert_f32_close(got, want, what: str, tol: float = REL_TOL, floor: float = RMS_FLOOR):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite values"
    e = floored_rel_err(got, want, floor)
    _record(kind="f32", what=what, n=int(np.size(want)), floored=e, floor=floor,
            elementwise=elementwise_rel_err(got, want))
    assert e <= tol, "%s: floored relative error %.3g > %.1g (floor %g * rms)" % (what, e, tol, floor)


def assert_product_close(got, want, s, u, what: str, tol: float = REL_TOL):
    """Outputs o = s * u of two f32 dot products (the FusedFFN's silu(gate) * up): the error of
    each factor is held to the section rule, so the product's is |s| du + |u| ds to first order
    and the floor of element i is RMS_FLOOR * (|s_i| rms(u) + rms(s) |u_i|) in place of a
    fraction of rms(o).  s and u are the oracle's factors (double)."""
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite values"
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    s = np.asarray(s, np.float64).ravel()
    u = np.asarray(u, np.float64).ravel()
    floor = RMS_FLOOR * (np.abs(s) * _rms(u) + _rms(s) * np.abs(u))
    e = float(np.max(np.abs(g - o) / np.maximum(np.abs(o), np.maximum(floor, 1e-30)))) if o.size else 0.0
    _record(kind="f32", what=what, n=int(o.size), floored=e, elementwise=elementwise_rel_err(got, want))
    assert e <= tol, "%s: floored relative error %.3g > %.1g (product floor)" % (what, e, tol)


def f16_ordered(codes) -> np.ndarray:
    c = np.asarray(codes, np.uint16).astype(np.int32)
    return np.where(c & 0x8000, -(c & 0x7FFF), c)


def f16_value(codes) -> np.ndarray:
    return np.asarray(codes, np.uint16).view(np.float16).astype(np.float64)


def f16_spacing(v) -> np.ndarray:
    """Distance from |v| to the next larger binary16 value (2^-24 in the subnormal range)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -24)))
    return np.ldexp(1.0, (np.maximum(e, -14) - 10).astype(np.int64))


def assert_f16_close(got_codes, want_codes, want_f32, what: str, rms: float | None = None,
                     floor: float = RMS_FLOOR):
    """f16 codes against the oracle's codes; want_f32 is the oracle's f32 value of each
    element (its magnitude decides the rule), rms the section's RMS (default: of want_f32),
    floor the f32 rule's floor for this output."""
    got_codes = np.asarray(got_codes, np.uint16).ravel()
    want_codes = np.asarray(want_codes, np.uint16).ravel()
    o = np.asarray(want_f32, np.float64).ravel()
    assert o.size == want_codes.size, (what, o.size, want_codes.size)
    rms = _rms(o) if rms is None else rms
    ulp = np.abs(f16_ordered(got_codes) - f16_ordered(want_codes))
    small = np.abs(o) < floor * rms
    diff = np.abs(f16_value(got_codes) - f16_value(want_codes))
    near = small & (diff <= REL_TOL * floor * rms + f16_spacing(o))
    ok = (ulp <= 1) | near
    via_floor = near & (ulp > 1)
    _record(kind="f16", what=what, n=int(o.size), max_ulp=int(ulp.max()) if ulp.size else 0,
            below_floor=int(small.sum()), accepted_via_floor=int(via_floor.sum()),
            max_ulp_via_floor=int(ulp[via_floor].max()) if via_floor.any() else 0,
            max_ulp_at_or_above_floor=int(ulp[~small].max()) if (~small).any() else 0)
    bad = ~ok
    assert not bad.any(), "%s: %d f16 values beyond the rule (max ulp %d, %d of them at or above %g * rms)" % (
        what, int(bad.sum()), int(ulp.max()), int((bad & ~small).sum()), floor)


def assert_kv_region(got, want, pos, what: str, section_f32=None, floor: float = RMS_FLOOR):
    """Rows != pos bit-identical; row pos within tolerance (f32) or the f16 rule.  For f16
    caches, section_f32 is the oracle's f32 values of the row (one row checked), else the
    oracle's f16 values stand in for them."""
    assert got.shape == want.shape and got.dtype == want.dtype, what
    gb = got.view(np.uint32 if got.dtype == np.float32 else np.uint16)
    wb = want.view(np.uint32 if want.dtype == np.float32 else np.uint16)
    mask = np.ones(got.shape[0], bool)
    if pos is not None:
        mask[list(np.atleast_1d(pos))] = False
    assert np.array_equal(gb[mask], wb[mask]), what + ": untouched rows changed"
    _record(kind="kv_untouched", what=what, rows=int(mask.sum()), bit_exact=True)
    if pos is None:
        return
    rows = list(np.atleast_1d(pos))
    for p in rows:
        if got.dtype == np.float32:
            assert_f32_close(got[p], want[p], "%s row %d" % (what, p), floor=floor)
        else:
            o32 = section_f32 if (section_f32 is not None and len(rows) == 1) else f16_value(want[p])
            assert_f16_close(got[p], want[p], o32, "%s row %d" % (what, p), floor=floor)


def parity_summary(records=None) -> str:
    """One line: the largest errors over every comparison recorded."""
    recs = RECORDS if records is None else records
    f32 = [r for r in recs if r["kind"] == "f32"]
    f16 = [r for r in recs if r["kind"] == "f16"]
    kvu = [r for r in recs if r["kind"] == "kv_untouched"]
    if not (f32 or f16 or kvu):
        return ""
    parts = []
    for fl in sorted({r.get("floor", RMS_FLOOR) for r in f32}):
        sec = [r for r in f32 if r.get("floor", RMS_FLOOR) == fl]
        worst = max(sec, key=lambda r: r["floored"])
        parts.append("%d f32 sections (%d values) at floor %g*rms: max floored err %.3g (gate %g; worst %s), "
                     "max elementwise err %.3g" % (len(sec), sum(r["n"] for r in sec), fl, worst["floored"], REL_TOL,
                                                   worst["what"], max(r["elementwise"] for r in sec)))
    if f16:
        parts.append("%d f16 rows (%d values): max ulp %d at or above the floor, %d values accepted only "
                     "below it (max ulp %d)" % (len(f16), sum(r["n"] for r in f16),
                                                max(r["max_ulp_at_or_above_floor"] for r in f16),
                                                sum(r["accepted_via_floor"] for r in f16),
                                                max(r["max_ulp_via_floor"] for r in f16)))
    if kvu:
        parts.append("%d cache regions with untouched rows bit-exact (%d rows)" % (len(kvu),
                                                                                 sum(r["rows"] for r in kvu)))
    return "parity: " + "; ".join(parts)


# ---------------------------------------------------------------- canaries

def canary(n_ctx: int, nkt: int, kv_dtype: str, salt: int = 0) -> np.ndarray:
    """Per-slot NaN-payload fill, so any stray write shows up bit-exactly."""
    n = n_ctx * nkt
    idx = np.arange(n, dtype=np.uint64) + np.uint64(salt * 7919)
    if kv_dtype == "f32":
        return (np.uint32(0x7F800001) + (idx % np.uint64(0x3FFFFF)).astype(np.uint32)).reshape(
            n_ctx, nkt).view(np.float32)
    return (np.uint16(0x7C01) + (idx % np.uint64(0x1FF)).astype(np.uint16)).reshape(n_ctx, nkt)


# ---------------------------------------------------------------- device transfer

def to_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    return torch.from_numpy(a).cuda()


def to_host(t, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


# ---------------------------------------------------------------- seeded layers

class HostLayer:
    """Seeded inputs of one layer: concat W (row-keyed), bias, and section views."""

    def __init__(self, H, nh, nkv, hd, w_dtype, layer, seed=0):
        self.H, self.nh, self.nkv, self.hd = H, nh, nkv, hd
        self.nqt, self.nkt = nh * hd, nkv * hd
        self.R = self.nqt + 2 * self.nkt
        self.W = synth.weight_rows(seed, layer, 0, self.R, H, w_dtype)
        self.bias = synth.bias(seed, layer, self.R)
        self.layer, self.seed = layer, seed

    def sections(self):
        a, b = self.nqt, self.nqt + self.nkt
        return self.W[:a], self.W[a:b], self.W[b:]

    def bias_sections(self):
        a, b = self.nqt, self.nqt + self.nkt
        return self.bias[:a], self.bias[a:b], self.bias[b:]

    def x(self, pos):
        return synth.hidden(self.seed, self.layer, pos, self.H)
