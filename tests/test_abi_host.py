"""Host-side checks of the C ABI (no GPU): the library loads, exports every entry
point include/qkv.h declares, validates arguments before touching CUDA, and its
size arithmetic matches the numbers printed on the pages."""
import ctypes
import os

import numpy as np
import pytest

import oracle_pins as pins
import qkv_rope_kv_gb300 as q
from qkv_rope_kv_gb300 import configs


@pytest.fixture(scope="module")
def lib():
    return q.load()


def _desc(**kw):
    base = dict(hidden=5120, n_head=40, n_head_kv=8, head_dim=128, theta=1e6, freq_scale=1.0,
                n_ctx=4096, w_dtype=q.QKV_BF16, kv_dtype=q.QKV_F16,
                layer_class=q.QKV_CLASS_CONCAT, rope=q.QKV_ROPE_NEOX)
    base.update(kw)
    return q.qkv_plan_desc(**base)


def _create(lib, d):
    h = ctypes.c_void_p()
    st = lib.qkv_plan_create(ctypes.byref(d), ctypes.byref(h))
    if st == 0:
        lib.qkv_plan_destroy(h)
    return st


def test_exports_every_declared_entry_point(lib):
    names = q.header_entry_points()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert lib.qkv_abi_version() == 1
    assert lib.qkv_status_str(3) == b"QKV_ERR_POS_RANGE"


@pytest.mark.parametrize("kw,status", [
    (dict(), q.QKV_OK),
    (dict(hidden=0), q.QKV_ERR_INVALID_ARG),
    (dict(n_head=0), q.QKV_ERR_INVALID_ARG),
    (dict(n_ctx=0), q.QKV_ERR_INVALID_ARG),
    (dict(theta=0.0), q.QKV_ERR_INVALID_ARG),
    (dict(theta=float("nan")), q.QKV_ERR_INVALID_ARG),
    (dict(freq_scale=-1.0), q.QKV_ERR_INVALID_ARG),
    (dict(layer_class=5), q.QKV_ERR_INVALID_ARG),
    (dict(rope=7), q.QKV_ERR_INVALID_ARG),
    (dict(rope=q.QKV_ROPE_INTERLEAVED), q.QKV_ERR_UNSUPPORTED),
    (dict(head_dim=127), q.QKV_ERR_UNSUPPORTED),
    (dict(head_dim=258), q.QKV_ERR_UNSUPPORTED),
    (dict(w_dtype=q.QKV_F16), q.QKV_ERR_UNSUPPORTED),
    (dict(kv_dtype=q.QKV_BF16), q.QKV_ERR_UNSUPPORTED),
    (dict(hidden=60000), q.QKV_ERR_UNSUPPORTED),
    (dict(hidden=7, head_dim=2, n_head=1, n_head_kv=1), q.QKV_OK),
])
def test_plan_validation(lib, kw, status):
    assert _create(lib, _desc(**kw)) == status


def test_plan_create_null_args(lib):
    h = ctypes.c_void_p()
    assert lib.qkv_plan_create(None, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG
    assert lib.qkv_plan_create(ctypes.byref(_desc()), None) == q.QKV_ERR_INVALID_ARG
    assert b"null" in lib.qkv_last_error()


def test_sizes_match_pages():
    shapes = {"qwen2.5-14b": configs.QWEN14B, "qwen2.5-7b": configs.QWEN7B}
    for row in pins.read_golden("pages_shapes.txt"):
        if row[0] == "units":
            w = shapes[row[1]]
            p = q.qkv_plan_create(w.hidden, w.n_head, w.n_head_kv, w.head_dim, w.theta, w.n_ctx)
            assert p.info.epilogue_units == int(row[2])
        elif row[0] == "concat_shape":
            w = shapes[row[1]]
            p = q.qkv_plan_create(w.hidden, w.n_head, w.n_head_kv, w.head_dim, w.theta, w.n_ctx)
            assert p.info.rows == int(row[2]) and w.hidden == int(row[3])
        elif row[0] == "kv_layer_bytes":
            nkt, n_ctx, total = (int(v) for v in row[2:5])
            p = q.qkv_plan_create(896, 14, 2, 64, 1e6, n_ctx, w_dtype=q.QKV_F32, kv_dtype=q.QKV_F32)
            assert p.info.nkt == nkt
            view = q.kv_cache_view(p, 0x1000, 0x2000)
            assert 2 * view.region_bytes == total
            assert view.row_stride_elems == nkt and view.k == 0x1000 and view.v == 0x2000
        elif row[0] == "ledger":
            # our launches per decode layer: one for both classes (page: 2 concat, 4 mixed)
            if row[1] in ("concat", "mixed"):
                p = q.qkv_plan_create(5120, 40, 8, 128, 1e6, 4096)
                assert p.info.launches_decode == 1 < int(row[2])


def test_algorithmic_bytes_match_workload_table():
    for w in (configs.QWEN05_SINGLE, configs.QWEN7B, configs.QWEN14B):
        p = q.qkv_plan_create(w.hidden, w.n_head, w.n_head_kv, w.head_dim, w.theta, w.n_ctx,
                              w_dtype=q.QKV_F32 if w.w_dtype == "f32" else q.QKV_BF16,
                              kv_dtype=q.QKV_F32 if w.kv_dtype == "f32" else q.QKV_F16)
        assert p.info.algo_bytes_decode == w.algo_bytes_per_layer()
    assert configs.QWEN14B.algo_bytes_per_layer() == 73_482_240
    assert configs.QWEN7B.algo_bytes_per_layer() == 33_083_392


def test_frequency_table_matches_oracle(orc):
    for (H, nh, nkv, hd, theta) in ((896, 14, 2, 64, 1e6), (5120, 40, 8, 128, 1e6), (64, 2, 1, 4, 1e4)):
        p = q.qkv_plan_create(H, nh, nkv, hd, theta, 16)
        assert np.array_equal(p.inv_freq().view(np.uint32),
                              orc.inv_freq_table(hd, theta, 1.0).view(np.uint32))


def test_null_pointers_rejected_before_cuda(lib):
    p = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16)
    with pytest.raises(q.QkvError) as e:
        q.qkv_decode_step(p, None, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == q.QKV_ERR_INVALID_ARG
    with pytest.raises(q.QkvError) as e:
        q.qkv_epilogue(p, 16, 16, 16, 16, 16, 16, None, 16, 16, stream=0)
    assert e.value.status == q.QKV_ERR_INVALID_ARG


def test_class_mismatch_rejected(lib):
    mixed = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16, layer_class=q.QKV_CLASS_MIXED)
    concat = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16)
    with pytest.raises(q.QkvError) as e:
        q.qkv_decode_step(mixed, 16, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == q.QKV_ERR_INVALID_ARG
    with pytest.raises(q.QkvError) as e:
        q.qkv_decode_step_mixed(concat, *([16] * 13), stream=0)
    assert e.value.status == q.QKV_ERR_INVALID_ARG


def test_prefill_guards(lib):
    f32 = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16, w_dtype=q.QKV_F32)
    with pytest.raises(q.QkvError) as e:
        q.qkv_prefill_step(f32, 16, 4, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == q.QKV_ERR_UNSUPPORTED
    mixed = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16, layer_class=q.QKV_CLASS_MIXED)
    with pytest.raises(q.QkvError) as e:
        q.qkv_prefill_step(mixed, 16, 4, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == q.QKV_ERR_UNSUPPORTED


def test_prefill_degenerate_token_counts(lib):
    """nt = 0 is a no-op that succeeds without touching the device; a negative nt is rejected;
    a head_dim the tensor-core tiles cannot pair (not a multiple of 64) is refused before any
    launch.  Stand-in addresses: nothing is dereferenced on these paths."""
    fake = 16 * 64
    bf16 = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16, w_dtype=q.QKV_BF16)
    q.qkv_prefill_step(bf16, fake, 0, fake, fake, fake, fake, fake, fake, stream=0)
    with pytest.raises(q.QkvError) as e:
        q.qkv_prefill_step(bf16, fake, -1, fake, fake, fake, fake, fake, fake, stream=0)
    assert e.value.status == q.QKV_ERR_INVALID_ARG
    with pytest.raises(q.QkvError) as e:
        q.qkv_prefill_step(bf16, fake, 3, fake, fake, fake, fake, fake, fake, stream=0)
    assert e.value.status == q.QKV_ERR_UNSUPPORTED
    assert b"multiple of 64" in lib.qkv_last_error()


def test_graph_create_guards(lib):
    p = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16)
    h = ctypes.c_void_p()
    plans = (ctypes.c_void_p * 1)(p.handle)
    layers = (q.qkv_layer_ptrs * 1)()
    assert lib.qkv_model_graph_create(plans, 0, layers, 16, 16, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG
    assert lib.qkv_model_graph_create(plans, 1, layers, 16, None, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG
    # layer 0 has null pointers: rejected before any capture starts
    assert lib.qkv_model_graph_create(plans, 1, layers, 16, 16, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG


def test_ffn_guards(lib):
    """FusedFFN arguments are validated on the host before any CUDA call."""
    f = lib.qkv_ffn_step
    ok = 16 * 64  # a 16-byte aligned stand-in address; nothing is dereferenced on failure
    assert f(0, 8, q.QKV_BF16, ok, ok, ok, None) == q.QKV_ERR_INVALID_ARG          # hidden < 1
    assert f(49160, 8, q.QKV_BF16, ok, ok, ok, None) == q.QKV_ERR_INVALID_ARG      # hidden > 49152
    assert f(64, 0, q.QKV_BF16, ok, ok, ok, None) == q.QKV_ERR_INVALID_ARG         # n_ff < 1
    assert f(64, 8, q.QKV_F16, ok, ok, ok, None) == q.QKV_ERR_INVALID_ARG          # f16 weights
    assert f(64, 8, q.QKV_BF16, None, ok, ok, None) == q.QKV_ERR_INVALID_ARG       # null x
    assert f(64, 8, q.QKV_BF16, ok + 4, ok, ok, None) == q.QKV_ERR_INVALID_ARG     # misaligned x
    assert f(64, 8, q.QKV_BF16, ok, ok + 8, ok, None) == q.QKV_ERR_INVALID_ARG     # misaligned weights
    assert f(12, 8, q.QKV_BF16, ok, ok, ok, None) == q.QKV_ERR_UNSUPPORTED         # 24-byte rows
    h = ctypes.c_void_p()
    layers = (q.qkv_ffn_layer * 1)()
    g = lib.qkv_ffn_graph_create
    assert g(64, 8, q.QKV_BF16, 0, layers, 16, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG
    assert g(64, 8, q.QKV_BF16, 1, layers, None, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG
    assert g(64, 8, q.QKV_BF16, 1, layers, 16, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG  # null layer 0


def test_rmsnorm_guards(lib):
    """The fused RMSNorm entry points validate the norm arguments on the host."""
    p = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16)
    for args in ((None, 1e-6), (16, -1.0), (16, float("nan"))):
        with pytest.raises(q.QkvError) as e:
            q.qkv_decode_step_rmsnorm(p, 16, args[0], args[1], 16, 16, 16, 16, 16, 16, 16, 16, stream=0)
        assert e.value.status == q.QKV_ERR_INVALID_ARG
    mixed = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16, layer_class=q.QKV_CLASS_MIXED)
    with pytest.raises(q.QkvError) as e:
        q.qkv_decode_step_rmsnorm(mixed, 16, 16, 1e-6, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == q.QKV_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    plans = (ctypes.c_void_p * 1)(p.handle)
    layers = (q.qkv_layer_ptrs * 1)()
    norms = (ctypes.c_void_p * 1)(None)
    g = lib.qkv_model_graph_create_rmsnorm
    assert g(plans, 1, layers, None, ctypes.c_float(1e-6), 16, 16, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG
    assert g(plans, 1, layers, norms, ctypes.c_float(1e-6), 16, 16, ctypes.byref(h)) == q.QKV_ERR_INVALID_ARG



def test_qknorm_guards(lib):
    """FusedQkvNorm arguments are validated on the host before any CUDA call."""
    fake = 16 * 64  # 16-byte aligned stand-in address; nothing is dereferenced on failure
    p = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16)
    assert q.qkv_qknorm_workspace_bytes(p) == 3 * 4
    f = lib.qkv_decode_step_qknorm
    args = [p.handle, fake, fake, fake, fake, fake, ctypes.c_float(1e-6), fake, fake, fake, fake, fake, fake, fake,
            None]
    for i, bad in ((4, None), (5, None), (13, None), (13, fake + 2)):
        a = list(args)
        a[i] = bad
        assert f(*a) == q.QKV_ERR_INVALID_ARG, i
    for eps in (-1.0, float("nan")):
        a = list(args)
        a[6] = ctypes.c_float(eps)
        assert f(*a) == q.QKV_ERR_INVALID_ARG
    a = list(args)
    a[1] = fake + 4  # x not 16-byte aligned: no ring form
    assert f(*a) == q.QKV_ERR_UNSUPPORTED
    mixed = q.qkv_plan_create(64, 2, 1, 8, 1e4, 16, layer_class=q.QKV_CLASS_MIXED)
    a = list(args)
    a[0] = mixed.handle
    assert f(*a) == q.QKV_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    plans = (ctypes.c_void_p * 1)(p.handle)
    layers = (q.qkv_layer_ptrs * 1)()
    for name, _ in q.qkv_layer_ptrs._fields_:
        setattr(layers[0], name, fake)
    norms = (ctypes.c_void_p * 1)(fake)
    g = lib.qkv_model_graph_create_qknorm
    assert g(plans, 1, layers, norms, norms, ctypes.c_float(1e-6), fake, None, fake, ctypes.byref(h)) == \
        q.QKV_ERR_INVALID_ARG
    assert g(plans, 1, layers, None, norms, ctypes.c_float(1e-6), fake, fake, fake, ctypes.byref(h)) == \
        q.QKV_ERR_INVALID_ARG
    assert g(plans, 0, layers, norms, norms, ctypes.c_float(1e-6), fake, fake, fake, ctypes.byref(h)) == \
        q.QKV_ERR_INVALID_ARG


def test_plan_free_entry_points_load_the_library():
    """Entry points that take no plan load libqkv.so themselves: in a fresh interpreter,
    null arguments come back as the library's own INVALID_ARG status."""
    import subprocess
    import sys
    code = ("import qkv_rope_kv_gb300 as Q\n"
            "for f, a in ((Q.qkv_chain_add_bias, (None, None, 1)),\n"
            "             (Q.qkv_ffn_step, (8, 4, Q.QKV_F32, None, None, None))):\n"
            "    try:\n"
            "        f(*a, stream=0)\n"
            "    except Q.QkvError as e:\n"
            "        assert e.status == Q.QKV_ERR_INVALID_ARG, e\n"
            "    else:\n"
            "        raise SystemExit('no error for null pointers')\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stdout + r.stderr


def _c_kind(decl: str) -> str:
    """Category of a C parameter or return type (without its name) as it crosses the ABI."""
    if "*" in decl:
        return "ptr"
    base = decl.replace("const", "").split()[0]
    return {"float": "f32", "int32_t": "i32", "int": "i32", "qkv_status": "i32", "int64_t": "i64",
            "size_t": "size", "void": "void", "uint32_t": "u32"}[base]


def _ctypes_kind(t) -> str:
    if t is None:
        return "void"
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    return {ctypes.c_float: "f32", ctypes.c_int32: "i32", ctypes.c_int64: "i64",
            ctypes.c_size_t: "size", ctypes.c_uint32: "u32"}[t]


def _signature_mismatches(lib):
    import re
    text = re.sub(r"/\*.*?\*/", "", "".join(open(h).read() for h in q.HEADERS), flags=re.S)
    protos = re.findall(r"\n([A-Za-z_][\w\s\*]*?)\b((?:qkv|kv)_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text)
    assert sorted(name for _, name, _ in protos) == q.header_entry_points()
    bad = []
    for ret, name, args in protos:
        # every parameter in the header is named: its type is all but the last token
        params = [] if args.strip() in ("", "void") else [a.strip().rsplit(None, 1)[0] for a in args.split(",")]
        want = ([_c_kind(t) for t in params], _c_kind(ret))
        fn = getattr(lib, name)
        got = ([_ctypes_kind(t) for t in (fn.argtypes or [])], _ctypes_kind(fn.restype))
        if got != want:
            bad.append((name, got, want))
    return bad


def test_binding_signatures_match_header(lib):
    """Every prototype in include/qkv.h and the ctypes declaration of the same name agree on
    the number of parameters, each one's kind (pointer, f32, 32/64-bit integer, size_t) and
    the return kind: a drifted declaration would pass garbage without an error."""
    assert _signature_mismatches(lib) == []


def test_wait_timeout_hook_guards(lib):
    """The failure-path test hook rejects a wait limit outside 1 .. 1000 us and null pointers
    before any CUDA call."""
    plan = q.qkv_plan_create(64, 2, 1, 32, 1e4, 4)
    fake = 16 * 64
    for us, want in ((0, q.QKV_ERR_INVALID_ARG), (1001, q.QKV_ERR_INVALID_ARG)):
        st = lib.qkv_test_decode_wait_timeout(plan.handle, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                              us, None)
        assert st == want and b"wait_limit_us" in lib.qkv_last_error()
    st = lib.qkv_test_decode_wait_timeout(plan.handle, None, fake, fake, fake, fake, fake, fake, fake, fake, 100,
                                          None)
    assert st == q.QKV_ERR_INVALID_ARG and b"x is null" in lib.qkv_last_error()


def test_prefill_xchg_timeout_hook_guards(lib):
    """The prefill failure-path hook rejects a wait limit outside 1 .. 1000 us, null pointers and
    a shape that does not run on clusters of 2 (an odd number of 64-row tiles), before any CUDA
    call."""
    fake = 16 * 64
    plan = q.qkv_plan_create(256, 4, 2, 64, 1e4, 8, w_dtype=q.QKV_BF16)  # R = 512: 8 tiles
    for us in (0, 1001):
        st = lib.qkv_test_prefill_xchg_timeout(plan.handle, fake, 4, fake, fake, fake, fake, fake, fake, us, None)
        assert st == q.QKV_ERR_INVALID_ARG and b"wait_limit_us" in lib.qkv_last_error()
    st = lib.qkv_test_prefill_xchg_timeout(plan.handle, None, 4, fake, fake, fake, fake, fake, fake, 100, None)
    assert st == q.QKV_ERR_INVALID_ARG and b"null pointer" in lib.qkv_last_error()
    odd = q.qkv_plan_create(256, 1, 1, 64, 1e4, 8, w_dtype=q.QKV_BF16)  # R = 192: 3 tiles
    st = lib.qkv_test_prefill_xchg_timeout(odd.handle, fake, 4, fake, fake, fake, fake, fake, fake, 100, None)
    assert st == q.QKV_ERR_UNSUPPORTED and b"clusters of 2" in lib.qkv_last_error()
