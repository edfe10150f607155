"""Helpers for the GPU parity tests: seeded layers, device transfer, comparison rules.

Comparison rules (the tolerance the stage's arithmetic supports):
  * cache addressing and untouched slots: bit-exact;
  * q / k / v and f32 cache values: |g - o| <= 1e-4 * max(|o|, rms(o)) per
    section, i.e. 1e-4 relative at or above the section's RMS and 1e-4 * RMS
    absolute below it, where f32 accumulation of H products cannot keep an
    elementwise relative bound near zero;
  * f16 cache values: the f16 code within 1 ulp of the oracle's code, or (for
    values the f32 rule already floors) within that f32 absolute bound.
"""
from __future__ import annotations

import numpy as np

from qkv_rope_kv_gb300 import synth

REL_TOL = 1e-4


# ---------------------------------------------------------------- comparison

def floored_rel_err(got, want) -> float:
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    if o.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(o * o)))
    den = np.maximum(np.abs(o), max(rms, 1e-30))
    return float(np.max(np.abs(g - o) / den))


def elementwise_rel_err(got, want) -> float:
    """Unfloored max |g-o|/|o| over |o| > 0 (reported, not gated)."""
    g = np.asarray(got, np.float64).ravel()
    o = np.asarray(want, np.float64).ravel()
    m = o != 0
    return float(np.max(np.abs(g[m] - o[m]) / np.abs(o[m]))) if m.any() else 0.0


def assert_f32_close(got, want, what: str, tol: float = REL_TOL):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite values"
    e = floored_rel_err(got, want)
    assert e <= tol, "%s: floored relative error %.3g > %.1g" % (what, e, tol)


def f16_ordered(codes) -> np.ndarray:
    c = np.asarray(codes, np.uint16).astype(np.int32)
    return np.where(c & 0x8000, -(c & 0x7FFF), c)


def f16_value(codes) -> np.ndarray:
    return np.asarray(codes, np.uint16).view(np.float16).astype(np.float64)


def assert_f16_close(got_codes, want_codes, want_f32_section, what: str):
    ulp = np.abs(f16_ordered(got_codes) - f16_ordered(want_codes))
    sec = np.asarray(want_f32_section, np.float64)
    rms = float(np.sqrt(np.mean(sec * sec))) if sec.size else 0.0
    near = np.abs(f16_value(got_codes) - f16_value(want_codes)) <= REL_TOL * rms
    bad = ~((ulp <= 1) | near)
    assert not bad.any(), "%s: %d f16 values beyond 1 ulp (max ulp %d)" % (what, int(bad.sum()), int(ulp.max()))


def assert_kv_region(got, want, pos, what: str, section_f32=None):
    """Rows != pos bit-identical; row pos within tolerance (f32) or 1 ulp (f16)."""
    assert got.shape == want.shape and got.dtype == want.dtype, what
    gb = got.view(np.uint32 if got.dtype == np.float32 else np.uint16)
    wb = want.view(np.uint32 if want.dtype == np.float32 else np.uint16)
    mask = np.ones(got.shape[0], bool)
    if pos is not None:
        mask[list(np.atleast_1d(pos))] = False
    assert np.array_equal(gb[mask], wb[mask]), what + ": untouched rows changed"
    if pos is None:
        return
    for p in np.atleast_1d(pos):
        if got.dtype == np.float32:
            assert_f32_close(got[p], want[p], "%s row %d" % (what, p))
        else:
            assert_f16_close(got[p], want[p], section_f32 if section_f32 is not None else f16_value(want[p]),
                             "%s row %d" % (what, p))


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
