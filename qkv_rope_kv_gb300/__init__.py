"""Python binding of libqkv.so: the decode attention-input stage on GB300.

Argument marshalling only.  Every step of the stage runs in the CUDA kernels
of ``libqkv.so`` (declared in ``include/qkv.h``); this module turns torch
tensors into device pointers and torch streams into ``cudaStream_t`` handles,
calls the C entry point of the same name, and raises ``QkvError`` on any
non-zero status.  There is no CPU fallback: if the library is missing the
first call raises.

torch is imported lazily, so ``qkv_rope_kv_gb300.synth`` stays importable
without it.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqkv.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "qkv.h")
# every header of the C ABI: the stage (qkv.h) and the test hook of its failure path (qkv_test.h)
HEADERS = (HEADER, os.path.join(os.path.dirname(_HERE), "include", "qkv_test.h"))

# ---- constants mirrored from include/qkv.h ----
QKV_OK, QKV_ERR_INVALID_ARG, QKV_ERR_UNSUPPORTED, QKV_ERR_POS_RANGE, QKV_ERR_CUDA, \
    QKV_ERR_DEVICE_FLAG = range(6)
QKV_F32, QKV_BF16, QKV_F16 = 0, 1, 2
QKV_CLASS_CONCAT, QKV_CLASS_MIXED = 0, 1
QKV_ROPE_NEOX, QKV_ROPE_INTERLEAVED = 0, 1
QKV_MAX_HEAD_DIM = 256


class QkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, str(status)), message))
        self.status = status


_STATUS_NAMES = {0: "QKV_OK", 1: "QKV_ERR_INVALID_ARG", 2: "QKV_ERR_UNSUPPORTED",
                 3: "QKV_ERR_POS_RANGE", 4: "QKV_ERR_CUDA", 5: "QKV_ERR_DEVICE_FLAG"}


class qkv_plan_desc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_head", ctypes.c_int32),
                ("n_head_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("theta", ctypes.c_float), ("freq_scale", ctypes.c_float),
                ("n_ctx", ctypes.c_int32), ("w_dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("layer_class", ctypes.c_int32),
                ("rope", ctypes.c_int32)]


class qkv_plan_info(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("nqt", ctypes.c_int64), ("nkt", ctypes.c_int64),
                ("pair_units", ctypes.c_int64), ("epilogue_units", ctypes.c_int64),
                ("weight_bytes", ctypes.c_int64), ("kv_row_bytes", ctypes.c_int64),
                ("kv_region_bytes", ctypes.c_int64), ("algo_bytes_decode", ctypes.c_int64),
                ("launches_decode", ctypes.c_int32), ("weight_vectorized", ctypes.c_int32)]


class qkv_kv_view(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("n_ctx", ctypes.c_int32), ("nkt", ctypes.c_int64),
                ("row_stride_elems", ctypes.c_int64), ("region_bytes", ctypes.c_int64)]


class qkv_layer_ptrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("x", "w", "wq", "wk", "wv", "bias", "bias_q", "bias_k", "bias_v", "q", "k", "v",
                 "kv_k", "kv_v")]


class qkv_prefill_ptrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("X", "w", "bias", "positions", "Y", "kv_k", "kv_v")]


class qkv_ffn_layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "w_gate_up", "out")]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libqkv.so (after torch, which provides the CUDA runtime)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        import torch  # noqa: F401  (loads libcudart before libqkv)
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise QkvError(QKV_ERR_CUDA, "libqkv.so not found at %s: build it with "
                           "`python -c \"import __graft_entry__ as g; g.build()\"`" % p)
        lib = ctypes.CDLL(p)
        _declare(lib)
        if path is None:
            _lib = lib
        return lib


def _declare(lib):
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    st = ctypes.c_int
    sig = {
        "qkv_abi_version": ([], ctypes.c_int),
        "qkv_status_str": ([st], ctypes.c_char_p),
        "qkv_last_error": ([], ctypes.c_char_p),
        "qkv_plan_create": ([ctypes.POINTER(qkv_plan_desc), ctypes.POINTER(vp)], st),
        "qkv_plan_destroy": ([vp], None),
        "qkv_plan_info_get": ([vp, ctypes.POINTER(qkv_plan_info)], st),
        "qkv_plan_inv_freq": ([vp, vp, i32], st),
        "qkv_decode_step": ([vp] * 10 + [vp], st),
        "qkv_decode_step_mixed": ([vp] * 15, st),
        "qkv_decode_step_rmsnorm": ([vp, vp, vp, ctypes.c_float] + [vp] * 9, st),
        "qkv_model_graph_create_rmsnorm": ([vp, i32, vp, vp, ctypes.c_float, vp, vp, ctypes.POINTER(vp)], st),
        "qkv_project": ([vp] * 9, st),
        "qkv_epilogue": ([vp] * 11, st),
        "qkv_chain_add_bias": ([vp, vp, i64, vp], st),
        "qkv_chain_rope": ([vp, vp, i32, vp, vp], st),
        "qkv_chain_store": ([vp, vp, vp, vp, vp], st),
        "qkv_prefill_step": ([vp, vp, i32, vp, vp, vp, vp, vp, vp, vp], st),
        "kv_cache_view": ([vp, vp, vp, ctypes.POINTER(qkv_kv_view)], st),
        "qkv_model_graph_create": ([vp, i32, vp, vp, vp, ctypes.POINTER(vp)], st),
        "qkv_model_graph_launch": ([vp, vp], st),
        "qkv_prefill_graph_create": ([vp, i32, vp, i32, vp, ctypes.POINTER(vp)], st),
        "qkv_ffn_step": ([i32, i32, i32, vp, vp, vp, vp], st),
        "qkv_ffn_graph_create": ([i32, i32, i32, i32, vp, vp, ctypes.POINTER(vp)], st),
        "qkv_model_graph_run_host": ([vp, vp, vp, sz, vp, vp, sz, vp], st),
        "qkv_model_graph_kernel_count": ([vp, ctypes.POINTER(i32)], st),
        "qkv_qknorm_workspace_bytes": ([vp, ctypes.POINTER(sz)], st),
        "qkv_decode_step_qknorm": ([vp, vp, vp, vp, vp, vp, ctypes.c_float] + [vp] * 8, st),
        "qkv_decode_step_qknorm_noalloc": ([vp, vp, vp, vp, vp, vp, ctypes.c_float] + [vp] * 7, st),
        "qkv_model_graph_create_qknorm": ([vp, i32, vp, vp, vp, ctypes.c_float, vp, vp, vp, ctypes.POINTER(vp)], st),
        "qkv_model_graph_destroy": ([vp], None),
        "qkv_check_device_error": ([vp, ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(i32)], st),
        "qkv_test_decode_wait_timeout": ([vp] * 10 + [ctypes.c_uint32, vp], st),
        "qkv_test_prefill_xchg_timeout": ([vp, vp, ctypes.c_int32] + [vp] * 6 + [ctypes.c_uint32, vp], st),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res


def header_entry_points(paths=HEADERS) -> list[str]:
    """Names of the functions the headers of include/ declare."""
    text = "".join(open(p).read() for p in ([paths] if isinstance(paths, str) else paths))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:qkv|kv)_[a-z0-9_]+)\s*\(", text)))


def _check(status: int):
    if status != QKV_OK:
        msg = _lib.qkv_last_error().decode() if _lib is not None else ""
        raise QkvError(status, msg)


def _ptr(t) -> int | None:
    """Device pointer of a CUDA tensor (or a raw int / None passed through)."""
    if t is None or isinstance(t, int):
        return t
    if not t.is_cuda:
        raise QkvError(QKV_ERR_INVALID_ARG, "expected a CUDA tensor, got one on %s" % t.device)
    return t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- plans

class Plan:
    """Owner of a ``qkv_plan*``; destroyed with the object."""

    def __init__(self, handle: int, desc: qkv_plan_desc):
        self.handle = handle
        self.desc = desc

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.qkv_plan_destroy(self.handle)
            self.handle = None

    @property
    def info(self) -> qkv_plan_info:
        out = qkv_plan_info()
        _check(_lib.qkv_plan_info_get(self.handle, ctypes.byref(out)))
        return out

    def inv_freq(self):
        import numpy as np
        n = self.desc.head_dim // 2
        out = np.empty(n, np.float32)
        _check(_lib.qkv_plan_inv_freq(self.handle, out.ctypes.data, n))
        return out


def qkv_plan_create(hidden: int, n_head: int, n_head_kv: int, head_dim: int, theta: float,
                    n_ctx: int, w_dtype: int = QKV_BF16, kv_dtype: int = QKV_F16,
                    layer_class: int = QKV_CLASS_CONCAT, rope: int = QKV_ROPE_NEOX,
                    freq_scale: float = 1.0) -> Plan:
    load()
    d = qkv_plan_desc(hidden, n_head, n_head_kv, head_dim, theta, freq_scale, n_ctx, w_dtype,
                      kv_dtype, layer_class, rope)
    h = ctypes.c_void_p()
    _check(_lib.qkv_plan_create(ctypes.byref(d), ctypes.byref(h)))
    return Plan(h.value, d)


# ---------------------------------------------------------------- decode

def qkv_decode_step(plan: Plan, x, w, bias, d_pos, q, k, v, kv_k, kv_v, stream=None):
    _check(_lib.qkv_decode_step(plan.handle, _ptr(x), _ptr(w), _ptr(bias), _ptr(d_pos), _ptr(q),
                                _ptr(k), _ptr(v), _ptr(kv_k), _ptr(kv_v), _stream(stream)))


def qkv_test_decode_wait_timeout(plan: Plan, x, w, bias, d_pos, q, k, v, kv_k, kv_v, wait_limit_us: int = 200,
                                 stream=None):
    """Test hook (include/qkv_test.h): qkv_decode_step with each CTA's last weight copy withheld
    and every wait limited to wait_limit_us, so the device status flag 2 gets set."""
    _check(_lib.qkv_test_decode_wait_timeout(plan.handle, _ptr(x), _ptr(w), _ptr(bias), _ptr(d_pos), _ptr(q),
                                             _ptr(k), _ptr(v), _ptr(kv_k), _ptr(kv_v), int(wait_limit_us),
                                             _stream(stream)))


def qkv_test_prefill_xchg_timeout(plan: Plan, X, nt: int, w, bias, d_positions, Y, kv_k, kv_v,
                                  wait_limit_us: int = 200, stream=None):
    """Test hook (include/qkv_test.h): qkv_prefill_step with the exchange of partial sums
    withheld and every wait limited to wait_limit_us, so the device status flag 2 gets set."""
    _check(_lib.qkv_test_prefill_xchg_timeout(plan.handle, _ptr(X), int(nt), _ptr(w), _ptr(bias),
                                              _ptr(d_positions), _ptr(Y), _ptr(kv_k), _ptr(kv_v),
                                              int(wait_limit_us), _stream(stream)))


def qkv_decode_step_rmsnorm(plan: Plan, h, norm_w, norm_eps: float, w, bias, d_pos, q, k, v, kv_k, kv_v,
                            stream=None):
    """qkv_decode_step on RMSNorm(h) with weight norm_w, the norm computed in the kernel."""
    _check(_lib.qkv_decode_step_rmsnorm(plan.handle, _ptr(h), _ptr(norm_w), float(norm_eps), _ptr(w), _ptr(bias),
                                        _ptr(d_pos), _ptr(q), _ptr(k), _ptr(v), _ptr(kv_k), _ptr(kv_v),
                                        _stream(stream)))


def qkv_decode_step_mixed(plan: Plan, x, wq, wk, wv, bias_q, bias_k, bias_v, d_pos, q, k, v,
                          kv_k, kv_v, stream=None):
    _check(_lib.qkv_decode_step_mixed(plan.handle, _ptr(x), _ptr(wq), _ptr(wk), _ptr(wv),
                                      _ptr(bias_q), _ptr(bias_k), _ptr(bias_v), _ptr(d_pos),
                                      _ptr(q), _ptr(k), _ptr(v), _ptr(kv_k), _ptr(kv_v),
                                      _stream(stream)))


def qkv_project(plan: Plan, x, wq, wk, wv, q, k, v, stream=None):
    _check(_lib.qkv_project(plan.handle, _ptr(x), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(q), _ptr(k),
                            _ptr(v), _stream(stream)))


def qkv_epilogue(plan: Plan, q, k, v, bias_q, bias_k, bias_v, d_pos, kv_k, kv_v, stream=None):
    _check(_lib.qkv_epilogue(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(bias_q), _ptr(bias_k),
                             _ptr(bias_v), _ptr(d_pos), _ptr(kv_k), _ptr(kv_v), _stream(stream)))


def qkv_chain_add_bias(y, b, n: int, stream=None):
    _check(load().qkv_chain_add_bias(_ptr(y), _ptr(b), n, _stream(stream)))


def qkv_chain_rope(plan: Plan, y, n_heads: int, d_pos, stream=None):
    _check(_lib.qkv_chain_rope(plan.handle, _ptr(y), n_heads, _ptr(d_pos), _stream(stream)))


def qkv_chain_store(plan: Plan, src, cache, d_pos, stream=None):
    _check(_lib.qkv_chain_store(plan.handle, _ptr(src), _ptr(cache), _ptr(d_pos), _stream(stream)))


# ---------------------------------------------------------------- prefill

def qkv_prefill_step(plan: Plan, X, nt: int, w, bias, d_positions, Y, kv_k, kv_v, stream=None):
    _check(_lib.qkv_prefill_step(plan.handle, _ptr(X), nt, _ptr(w), _ptr(bias), _ptr(d_positions),
                                 _ptr(Y), _ptr(kv_k), _ptr(kv_v), _stream(stream)))


# ---------------------------------------------------------------- cache view

def kv_cache_view(plan: Plan, kv_k, kv_v) -> qkv_kv_view:
    out = qkv_kv_view()
    _check(_lib.kv_cache_view(plan.handle, _ptr(kv_k), _ptr(kv_v), ctypes.byref(out)))
    return out


# ---------------------------------------------------------------- model graph

class ModelGraph:
    """Owner of a ``qkv_graph*`` plus references keeping its plans and buffers alive."""

    def __init__(self, handle: int, keep):
        self.handle = handle
        self._keep = keep

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.qkv_model_graph_destroy(self.handle)
            self.handle = None

    def launch(self, stream=None):
        _check(_lib.qkv_model_graph_launch(self.handle, _stream(stream)))

    def run_host(self, h_in, d_in, d_out, h_out, stream=None):
        """Copy h_in -> d_in, replay, copy d_out -> h_out (host tensors should be pinned)."""
        in_bytes = 0 if h_in is None else h_in.numel() * h_in.element_size()
        out_bytes = 0 if h_out is None else h_out.numel() * h_out.element_size()
        _check(_lib.qkv_model_graph_run_host(
            self.handle, None if h_in is None else h_in.data_ptr(), _ptr(d_in), in_bytes,
            _ptr(d_out), None if h_out is None else h_out.data_ptr(), out_bytes, _stream(stream)))

    @property
    def kernel_count(self) -> int:
        out = ctypes.c_int32()
        _check(_lib.qkv_model_graph_kernel_count(self.handle, ctypes.byref(out)))
        return out.value


def qkv_model_graph_create(plans, layers, d_pos, stream) -> ModelGraph:
    """``layers``: list of dicts with the qkv_layer_ptrs field names -> tensors."""
    n = len(plans)
    assert len(layers) == n
    arr_plans = (ctypes.c_void_p * n)(*[p.handle for p in plans])
    arr_layers = (qkv_layer_ptrs * n)()
    for i, L in enumerate(layers):
        for name, _ in qkv_layer_ptrs._fields_:
            setattr(arr_layers[i], name, _ptr(L.get(name)))
    h = ctypes.c_void_p()
    _check(_lib.qkv_model_graph_create(arr_plans, n, arr_layers, _ptr(d_pos), _stream(stream),
                                       ctypes.byref(h)))
    return ModelGraph(h.value, (plans, layers, d_pos))


def qkv_model_graph_create_rmsnorm(plans, layers, norm_w, norm_eps: float, d_pos, stream) -> ModelGraph:
    """As qkv_model_graph_create with each layer's RMSNorm fused in front: layers[i]["x"] is
    the hidden state before the norm, norm_w[i] the layer's norm weight (device tensors)."""
    n = len(plans)
    assert len(layers) == n and len(norm_w) == n
    arr_plans = (ctypes.c_void_p * n)(*[p.handle for p in plans])
    arr_layers = (qkv_layer_ptrs * n)()
    for i, L in enumerate(layers):
        for name, _ in qkv_layer_ptrs._fields_:
            setattr(arr_layers[i], name, _ptr(L.get(name)))
    arr_norm = (ctypes.c_void_p * n)(*[_ptr(t) for t in norm_w])
    h = ctypes.c_void_p()
    _check(_lib.qkv_model_graph_create_rmsnorm(arr_plans, n, arr_layers, arr_norm, float(norm_eps), _ptr(d_pos),
                                               _stream(stream), ctypes.byref(h)))
    return ModelGraph(h.value, (plans, layers, norm_w, d_pos))


def qkv_qknorm_workspace_bytes(plan: Plan) -> int:
    out = ctypes.c_size_t()
    _check(_lib.qkv_qknorm_workspace_bytes(plan.handle, ctypes.byref(out)))
    return out.value


def qkv_decode_step_qknorm(plan: Plan, x, w, bias, q_norm_w, k_norm_w, eps: float, d_pos, q, k, v, kv_k, kv_v,
                           workspace, stream=None):
    """qkv_decode_step with per-head q/k RMSNorm (FusedQkvNorm); ``workspace`` is a zeroed device
    buffer of qkv_qknorm_workspace_bytes(plan) bytes, left zeroed."""
    _check(_lib.qkv_decode_step_qknorm(plan.handle, _ptr(x), _ptr(w), _ptr(bias), _ptr(q_norm_w), _ptr(k_norm_w),
                                       float(eps), _ptr(d_pos), _ptr(q), _ptr(k), _ptr(v), _ptr(kv_k), _ptr(kv_v),
                                       _ptr(workspace), _stream(stream)))


def qkv_decode_step_qknorm_noalloc(plan: Plan, x, w, bias, q_norm_w, k_norm_w, eps: float, d_pos, q, k, v, kv_k,
                                   kv_v, stream=None):
    """qkv_decode_step_qknorm without a workspace: the counters are the library's own fixed
    device array (at most 1024 q + kv heads; calls sharing it must not overlap on the GPU)."""
    _check(_lib.qkv_decode_step_qknorm_noalloc(plan.handle, _ptr(x), _ptr(w), _ptr(bias), _ptr(q_norm_w),
                                               _ptr(k_norm_w), float(eps), _ptr(d_pos), _ptr(q), _ptr(k), _ptr(v),
                                               _ptr(kv_k), _ptr(kv_v), _stream(stream)))


def qkv_model_graph_create_qknorm(plans, layers, q_norm_w, k_norm_w, eps: float, d_pos, workspace,
                                  stream) -> ModelGraph:
    """The FusedQkvNorm model graph: q_norm_w[i] / k_norm_w[i] per layer, one shared workspace."""
    n = len(plans)
    assert len(layers) == n and len(q_norm_w) == n and len(k_norm_w) == n
    arr_plans = (ctypes.c_void_p * n)(*[p.handle for p in plans])
    arr_layers = (qkv_layer_ptrs * n)()
    for i, L in enumerate(layers):
        for name, _ in qkv_layer_ptrs._fields_:
            setattr(arr_layers[i], name, _ptr(L.get(name)))
    arr_q = (ctypes.c_void_p * n)(*[_ptr(t) for t in q_norm_w])
    arr_k = (ctypes.c_void_p * n)(*[_ptr(t) for t in k_norm_w])
    h = ctypes.c_void_p()
    _check(_lib.qkv_model_graph_create_qknorm(arr_plans, n, arr_layers, arr_q, arr_k, float(eps), _ptr(d_pos),
                                              _ptr(workspace), _stream(stream), ctypes.byref(h)))
    return ModelGraph(h.value, (plans, layers, q_norm_w, k_norm_w, d_pos, workspace))


def qkv_prefill_graph_create(plans, layers, nt: int, stream) -> ModelGraph:
    """``layers``: list of dicts with the qkv_prefill_ptrs field names -> tensors."""
    n = len(plans)
    assert len(layers) == n
    arr_plans = (ctypes.c_void_p * n)(*[p.handle for p in plans])
    arr_layers = (qkv_prefill_ptrs * n)()
    for i, L in enumerate(layers):
        for name, _ in qkv_prefill_ptrs._fields_:
            setattr(arr_layers[i], name, _ptr(L.get(name)))
    h = ctypes.c_void_p()
    _check(_lib.qkv_prefill_graph_create(arr_plans, n, arr_layers, nt, _stream(stream), ctypes.byref(h)))
    return ModelGraph(h.value, (plans, layers))


# ---------------------------------------------------------------- FusedFFN

def qkv_ffn_step(hidden: int, n_ff: int, w_dtype: int, x, w_gate_up, out, stream=None):
    """out[i] = silu(g_i) * u_i over the concat gate|up weight (device tensors)."""
    _check(load().qkv_ffn_step(hidden, n_ff, w_dtype, _ptr(x), _ptr(w_gate_up), _ptr(out), _stream(stream)))


def qkv_ffn_graph_create(hidden: int, n_ff: int, w_dtype: int, layers, stream) -> ModelGraph:
    """``layers``: list of dicts with the qkv_ffn_layer field names -> tensors."""
    n = len(layers)
    arr = (qkv_ffn_layer * n)()
    for i, L in enumerate(layers):
        for name, _ in qkv_ffn_layer._fields_:
            setattr(arr[i], name, _ptr(L.get(name)))
    h = ctypes.c_void_p()
    _check(load().qkv_ffn_graph_create(hidden, n_ff, w_dtype, n, arr, _stream(stream), ctypes.byref(h)))
    return ModelGraph(h.value, (layers,))


# ---------------------------------------------------------------- device status

def qkv_check_device_error(stream=None, raise_on_flag: bool = False):
    """Return (flags, bad_pos) and clear the device status word."""
    flags = ctypes.c_uint32()
    bad = ctypes.c_int32()
    st = load().qkv_check_device_error(_stream(stream), ctypes.byref(flags), ctypes.byref(bad))
    if st not in (QKV_OK, QKV_ERR_DEVICE_FLAG) or (raise_on_flag and st != QKV_OK):
        _check(st)
    return flags.value, bad.value
