"""CPU oracle for the decode QKV stage — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library
and its Python binding) never imports, links or calls it.

The arithmetic lives in ``qkv_oracle.c`` (plain C, double precision, plain
loops); this module compiles it with gcc and exposes it through ctypes with
numpy arrays.  Every function's source comment cites the page passage it
follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qkv_oracle.c")
_LIB = os.path.join(_HERE, "libqkv_oracle.so")

OK = 0
POS_RANGE = 1
BAD_ARG = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB, defines=()) -> str:
    """Compile the oracle (no FMA contraction, so results match on x86 and Arm)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, src, "-lm"]
        cmd[1:1] = ["-D%s" % d for d in defines]
        subprocess.check_call(cmd)
        os.replace(tmp, out)
    return out


def _bind(lib):
    vp, i, i64, d, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = d
    lib.oracle_f32_to_f16.argtypes = [f]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_inv_freq.argtypes = [i, i, d, d]
    lib.oracle_inv_freq.restype = f
    lib.oracle_inv_freq_table.argtypes = [i, d, d, vp]
    lib.oracle_theta.argtypes = [i, f]
    lib.oracle_theta.restype = f
    lib.oracle_matvec.argtypes = [vp, i, vp, i64, i64, vp]
    lib.oracle_rope_pair.argtypes = [d, d, f, f, i, f, vp, vp]
    lib.oracle_qkv_token.argtypes = [vp, vp, i, i, i, d, d, i, i, i, vp, vp, vp, vp, vp]
    lib.oracle_qkv_token.restype = i
    lib.oracle_qkv_decode.argtypes = [vp, i, vp, vp, i, i, i, i, d, d, i, i, i, vp, vp, vp, vp,
                                      vp, vp]
    lib.oracle_qkv_decode.restype = i
    lib.oracle_qkv_decode_mixed.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, i, d, d, i, i, i, vp,
                                            vp, vp, vp, vp, vp]
    lib.oracle_qkv_decode_mixed.restype = i
    lib.oracle_qkv_prefill.argtypes = [vp, i, vp, i, vp, vp, i, i, i, i, d, d, i, i, vp, vp, vp,
                                       vp, vp]
    lib.oracle_qkv_prefill.restype = i
    lib.oracle_silu.argtypes = [d]
    lib.oracle_silu.restype = d
    lib.oracle_ffn_swiglu.argtypes = [vp, i, vp, i64, i64, vp]
    lib.oracle_rmsnorm.argtypes = [vp, vp, i64, d, vp]
    lib.oracle_qkv_token_qknorm.argtypes = [vp, vp, vp, vp, d, i, i, i, d, d, i, i, i, vp, vp, vp, vp, vp]
    lib.oracle_qkv_token_qknorm.restype = i
    lib.oracle_qkv_decode_qknorm.argtypes = [vp, i, vp, vp, vp, vp, d, i, i, i, i, d, d, i, i, i, vp, vp, vp,
                                             vp, vp, vp]
    lib.oracle_qkv_decode_qknorm.restype = i
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads a variant build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data


class Oracle:
    """numpy front end over one build of the oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    # scalar pieces
    def f32_to_f16(self, v: float) -> int:
        return int(self.lib.oracle_f32_to_f16(float(np.float32(v))))

    def inv_freq(self, d: int, hd: int, base: float, freq_scale: float = 1.0) -> np.float32:
        return np.float32(self.lib.oracle_inv_freq(d, hd, base, freq_scale))

    def inv_freq_table(self, hd: int, base: float, freq_scale: float = 1.0) -> np.ndarray:
        out = np.empty(hd // 2, dtype=np.float32)
        self.lib.oracle_inv_freq_table(hd, base, freq_scale, _p(out))
        return out

    def theta(self, pos: int, inv_freq: float) -> np.float32:
        return np.float32(self.lib.oracle_theta(pos, float(np.float32(inv_freq))))

    def rope_pair(self, y0, y1, b0, b1, pos, inv_freq):
        r0, r1 = ctypes.c_float(), ctypes.c_float()
        self.lib.oracle_rope_pair(float(y0), float(y1), float(b0), float(b1), int(pos),
                                  float(np.float32(inv_freq)), ctypes.byref(r0), ctypes.byref(r1))
        return np.float32(r0.value), np.float32(r1.value)

    def matvec(self, W: np.ndarray, x: np.ndarray) -> np.ndarray:
        """y = W x in double; W float32 [R, H] or uint16 bf16 bits [R, H]."""
        W = np.ascontiguousarray(W)
        x = np.ascontiguousarray(x, dtype=np.float32)
        R, H = W.shape
        y = np.empty(R, dtype=np.float64)
        self.lib.oracle_matvec(_p(W), int(W.dtype == np.uint16), _p(x), R, H, _p(y))
        return y

    def silu(self, v: float) -> float:
        return float(self.lib.oracle_silu(float(v)))

    def ffn_swiglu(self, W: np.ndarray, x: np.ndarray) -> np.ndarray:
        """silu(gate) * up over a concat gate|up weight W [2 nf, H] (float32 or bf16 bits)."""
        W = np.ascontiguousarray(W)
        x = np.ascontiguousarray(x, dtype=np.float32)
        R, H = W.shape
        assert R % 2 == 0, "the gate|up weight has 2 nf rows"
        out = np.empty(R // 2, dtype=np.float32)
        self.lib.oracle_ffn_swiglu(_p(W), int(W.dtype == np.uint16), _p(x), R // 2, H, _p(out))
        return out

    def rmsnorm(self, h: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
        """x = h * w / sqrt(mean(h^2) + eps), float32 out."""
        h = np.ascontiguousarray(h, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.float32)
        assert h.shape == w.shape and h.ndim == 1
        x = np.empty_like(h)
        self.lib.oracle_rmsnorm(_p(h), _p(w), h.size, float(eps), _p(x))
        return x

    def token(self, y, bias, nh, nkv, hd, base, freq_scale, pos, kv_k, kv_v):
        """Epilogue for one token on a precomputed projection y (float64 [R])."""
        nqt, nkt = nh * hd, nkv * hd
        q = np.empty(nqt, np.float32)
        k = np.empty(nkt, np.float32)
        v = np.empty(nkt, np.float32)
        n_ctx, f16 = _kv_meta(kv_k, kv_v, nkt)
        st = self.lib.oracle_qkv_token(_p(np.ascontiguousarray(y, np.float64)),
                                       _p(np.ascontiguousarray(bias, np.float32)), nh, nkv, hd,
                                       base, freq_scale, pos, n_ctx, f16, _p(q), _p(k), _p(v),
                                       _p(kv_k), _p(kv_v))
        return st, q, k, v

    def token_qknorm(self, y, bias, q_norm_w, k_norm_w, eps, nh, nkv, hd, base, freq_scale, pos, kv_k, kv_v):
        """FusedQkvNorm epilogue for one token on a precomputed projection y (float64 [R])."""
        nqt, nkt = nh * hd, nkv * hd
        q = np.empty(nqt, np.float32)
        k = np.empty(nkt, np.float32)
        v = np.empty(nkt, np.float32)
        n_ctx, f16 = _kv_meta(kv_k, kv_v, nkt)
        st = self.lib.oracle_qkv_token_qknorm(_p(np.ascontiguousarray(y, np.float64)),
                                              _p(np.ascontiguousarray(bias, np.float32)),
                                              _p(np.ascontiguousarray(q_norm_w, np.float32)),
                                              _p(np.ascontiguousarray(k_norm_w, np.float32)), float(eps), nh, nkv,
                                              hd, base, freq_scale, pos, n_ctx, f16, _p(q), _p(k), _p(v),
                                              _p(kv_k), _p(kv_v))
        return st, q, k, v

    def decode_qknorm(self, W, x, bias, q_norm_w, k_norm_w, eps, nh, nkv, hd, base, freq_scale, pos, kv_k, kv_v):
        """Concat-class FusedQkvNorm: projection, bias, per-head q/k RMSNorm (weights of hd values),
        neox RoPE, KV store.  kv_k/kv_v updated in place as in decode()."""
        nqt, nkt = nh * hd, nkv * hd
        R = nqt + 2 * nkt
        W = np.ascontiguousarray(W)
        assert W.shape[0] == R
        assert len(q_norm_w) == hd and len(k_norm_w) == hd
        y = np.full(R, np.nan)  # a row the oracle fails to compute shows up as NaN
        q = np.empty(nqt, np.float32)
        k = np.empty(nkt, np.float32)
        v = np.empty(nkt, np.float32)
        n_ctx, f16 = _kv_meta(kv_k, kv_v, nkt)
        st = self.lib.oracle_qkv_decode_qknorm(_p(W), int(W.dtype == np.uint16),
                                               _p(np.ascontiguousarray(x, np.float32)),
                                               _p(np.ascontiguousarray(bias, np.float32)),
                                               _p(np.ascontiguousarray(q_norm_w, np.float32)),
                                               _p(np.ascontiguousarray(k_norm_w, np.float32)), float(eps),
                                               W.shape[1], nh, nkv, hd, base, freq_scale, pos, n_ctx, f16, _p(y),
                                               _p(q), _p(k), _p(v), _p(kv_k), _p(kv_v))
        return st, q, k, v

    def decode(self, W, x, bias, nh, nkv, hd, base, freq_scale, pos, kv_k, kv_v):
        """Concat class. kv_k/kv_v: float32 or uint16 (f16 bits) arrays [n_ctx, nkt], updated in place."""
        nqt, nkt = nh * hd, nkv * hd
        R = nqt + 2 * nkt
        W = np.ascontiguousarray(W)
        assert W.shape[0] == R
        H = W.shape[1]
        y = np.full(R, np.nan)  # a row the oracle fails to compute shows up as NaN
        q = np.empty(nqt, np.float32)
        k = np.empty(nkt, np.float32)
        v = np.empty(nkt, np.float32)
        n_ctx, f16 = _kv_meta(kv_k, kv_v, nkt)
        st = self.lib.oracle_qkv_decode(_p(W), int(W.dtype == np.uint16),
                                        _p(np.ascontiguousarray(x, np.float32)),
                                        _p(np.ascontiguousarray(bias, np.float32)), H, nh, nkv,
                                        hd, base, freq_scale, pos, n_ctx, f16, _p(y), _p(q),
                                        _p(k), _p(v), _p(kv_k), _p(kv_v))
        return st, q, k, v

    def decode_mixed(self, Wq, Wk, Wv, x, bias, nh, nkv, hd, base, freq_scale, pos, kv_k, kv_v):
        nqt, nkt = nh * hd, nkv * hd
        Wq, Wk, Wv = (np.ascontiguousarray(a) for a in (Wq, Wk, Wv))
        assert Wq.dtype == Wk.dtype == Wv.dtype
        H = Wq.shape[1]
        y = np.full(nqt + 2 * nkt, np.nan)  # a row the oracle fails to compute shows up as NaN
        q = np.empty(nqt, np.float32)
        k = np.empty(nkt, np.float32)
        v = np.empty(nkt, np.float32)
        n_ctx, f16 = _kv_meta(kv_k, kv_v, nkt)
        st = self.lib.oracle_qkv_decode_mixed(_p(Wq), _p(Wk), _p(Wv), int(Wq.dtype == np.uint16),
                                              _p(np.ascontiguousarray(x, np.float32)),
                                              _p(np.ascontiguousarray(bias, np.float32)), H, nh,
                                              nkv, hd, base, freq_scale, pos, n_ctx, f16, _p(y),
                                              _p(q), _p(k), _p(v), _p(kv_k), _p(kv_v))
        return st, q, k, v

    def prefill(self, X_bf16, W, bias, positions, nh, nkv, hd, base, freq_scale, kv_k, kv_v):
        nqt, nkt = nh * hd, nkv * hd
        R = nqt + 2 * nkt
        X_bf16 = np.ascontiguousarray(X_bf16, np.uint16)
        W = np.ascontiguousarray(W)
        nt, H = X_bf16.shape
        positions = np.ascontiguousarray(positions, np.int32)
        xs = np.empty(H, np.float32)
        ys = np.full(R, np.nan)
        Y = np.empty((nt, R), np.float32)
        n_ctx, f16 = _kv_meta(kv_k, kv_v, nkt)
        st = self.lib.oracle_qkv_prefill(_p(X_bf16), nt, _p(W), int(W.dtype == np.uint16),
                                         _p(np.ascontiguousarray(bias, np.float32)),
                                         _p(positions), H, nh, nkv, hd, base, freq_scale, n_ctx,
                                         f16, _p(xs), _p(ys), _p(Y), _p(kv_k), _p(kv_v))
        return st, Y


def _kv_meta(kv_k: np.ndarray, kv_v: np.ndarray, nkt: int):
    assert kv_k.shape == kv_v.shape and kv_k.dtype == kv_v.dtype
    assert kv_k.flags.c_contiguous and kv_v.flags.c_contiguous
    assert kv_k.ndim == 2 and kv_k.shape[1] == nkt
    if kv_k.dtype == np.float32:
        return kv_k.shape[0], 0
    if kv_k.dtype == np.uint16:
        return kv_k.shape[0], 1
    raise TypeError("KV regions must be float32 or uint16 (f16 bit patterns)")
