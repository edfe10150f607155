"""Seeded synthetic inputs (weights, bias, hidden vectors) for the QKV stage.

This module only makes inputs; it contains none of the stage's arithmetic.
Both the CUDA path (benchmark, GPU tests) and the CPU oracle draw their
inputs from here, so the two sides see identical bytes without sharing any
compute code.

The generator is counter-based SplitMix64 with Box-Muller normals, written in
C (``synth.c``) so that multi-gigabyte weight sets are produced in seconds on
the host cores.  Every (tensor, layer, row-or-position) has its own stream.
Weight matrices are keyed per row of the concatenated ``wq|wk|wv`` layout, so
a separately generated ``wq``/``wk``/``wv`` block is bit-identical to the
matching rows of the concatenated matrix.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libqkv_synth.so")

# Stream tags.  Fixed forever: changing one changes every generated input.
T_WEIGHT = 1      # concat wq|wk|wv rows, keyed by global row index
T_BIAS = 2        # concat bq|bk|bv, keyed by index 0
T_HIDDEN = 3      # decode hidden vector x, keyed by position
T_PREFILL_X = 4   # prefill activations X[t], keyed by token index t
T_CANARY = 5      # KV-cache fill pattern for untouched-slot checks
T_FFN_WEIGHT = 6  # concat w_gate|w_up rows of the FFN, keyed by global row index
T_NORM = 7        # RMSNorm weight of the attention input, per layer

W_SIGMA = 0.02
BIAS_SIGMA = 0.1
X_SIGMA = 1.0
NORM_SIGMA = 0.1  # spread of the RMSNorm weight around 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libqkv_synth.so`` with gcc (OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, u32, i64, dbl = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_splitmix64.argtypes = [u64, u64]
            lib.synth_splitmix64.restype = u64
            lib.synth_stream_key.argtypes = [u64, u32, u32, u32]
            lib.synth_stream_key.restype = u64
            lib.synth_normal_at.argtypes = [u64, u64]
            lib.synth_normal_at.restype = dbl
            lib.synth_normal_f32.argtypes = [u64, u32, u32, u32, i64, dbl, vp]
            lib.synth_rows_f32.argtypes = [u64, u32, u32, i64, i64, i64, dbl, vp]
            lib.synth_rows_bf16.argtypes = [u64, u32, u32, i64, i64, i64, dbl, vp]
            lib.synth_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def splitmix64(state: int, n: int) -> int:
    """n-th output (n >= 1) of SplitMix64 started at ``state``."""
    return int(_load().synth_splitmix64(state, n))


def stream_key(seed: int, tensor: int, layer: int, index: int) -> int:
    return int(_load().synth_stream_key(seed, tensor, layer, index))


def normal_at(key: int, i: int) -> float:
    return float(_load().synth_normal_at(key, i))


def num_threads() -> int:
    return int(_load().synth_num_threads())


def normal_f32(seed: int, tensor: int, layer: int, index: int, n: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(seed, tensor, layer, index, n, sigma, out.ctypes.data)
    return out


def rows(seed: int, tensor: int, layer: int, row0: int, nrows: int, ncols: int, sigma: float,
         dtype: str, out: np.ndarray | None = None) -> np.ndarray:
    """Row-keyed matrix block; ``dtype`` is "f32" (float32) or "bf16" (uint16 bit patterns)."""
    if dtype == "f32":
        npdt, fn = np.float32, _load().synth_rows_f32
    elif dtype == "bf16":
        npdt, fn = np.uint16, _load().synth_rows_bf16
    else:
        raise ValueError("dtype must be 'f32' or 'bf16'")
    if out is None:
        out = np.empty((nrows, ncols), dtype=npdt)
    assert out.dtype == npdt and out.flags.c_contiguous and out.size == nrows * ncols
    fn(seed, tensor, layer, row0, nrows, ncols, sigma, out.ctypes.data)
    return out


# ---- workload-level helpers (the recipe used by tests and the benchmark) ----

def weight_rows(seed: int, layer: int, row0: int, nrows: int, hidden: int, dtype: str,
                out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+nrows) of the concatenated wq|wk|wv matrix, ~N(0, 0.02)."""
    return rows(seed, T_WEIGHT, layer, row0, nrows, hidden, W_SIGMA, dtype, out)


def ffn_weight_rows(seed: int, layer: int, row0: int, nrows: int, hidden: int, dtype: str,
                    out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+nrows) of the concatenated w_gate|w_up matrix, ~N(0, 0.02)."""
    return rows(seed, T_FFN_WEIGHT, layer, row0, nrows, hidden, W_SIGMA, dtype, out)


def norm_weight(seed: int, layer: int, h: int) -> np.ndarray:
    """RMSNorm weight of a layer, float32, 1 + N(0, 0.1)."""
    return (np.float32(1.0) + normal_f32(seed, T_NORM, layer, 0, h, NORM_SIGMA)).astype(np.float32)


def qk_norm_weights(seed: int, layer: int, hd: int):
    """Per-head q and k norm weights of a layer (hd values each, 1 + N(0, 0.1)): the
    norm-weight streams 1000 + 2 layer and 1001 + 2 layer."""
    return norm_weight(seed, 1000 + 2 * layer, hd), norm_weight(seed, 1001 + 2 * layer, hd)


def bias(seed: int, layer: int, n_rows: int) -> np.ndarray:
    """Concatenated bq|bk|bv, float32, ~N(0, 0.1)."""
    return normal_f32(seed, T_BIAS, layer, 0, n_rows, BIAS_SIGMA)


def hidden(seed: int, layer: int, pos: int, h: int) -> np.ndarray:
    """Decode input x for (layer, pos), float32, ~N(0, 1)."""
    return normal_f32(seed, T_HIDDEN, layer, pos, h, X_SIGMA)


def prefill_x(seed: int, layer: int, nt: int, h: int) -> np.ndarray:
    """Prefill activations X[nt, h] as bf16 bit patterns, ~N(0, 1), row t keyed by t."""
    return rows(seed, T_PREFILL_X, layer, 0, nt, h, X_SIGMA, "bf16")

