"""FusedFFN decode on the GPU against the oracle: out[i] = silu(gate_i) * up_i over a
concat gate|up weight (page "06 · Assign + fusion — every node picks an engine, then
patterns fold", §2.2-2.3), element by element at the FFN shapes of Qwen2.5-0.5B (f32),
7B and 14B (bf16) and at small ragged ones; the PDL-chained graph against sequential
steps, bitwise; and the whole-model graphs the FFN workloads time (24, 28 and 48
layers), every layer against the oracle."""
import numpy as np
import pytest

from gpu_helpers import assert_product_close, to_dev, to_host
from qkv_rope_kv_gb300 import configs, synth

pytestmark = pytest.mark.gpu

SEED = 0

SHAPES = [
    # H, nf, w dtype
    (896, 4864, "f32"),      # Qwen2.5-0.5B MLP (f32 weights)
    (3584, 18944, "bf16"),   # Qwen2.5-7B MLP
    (5120, 13824, "bf16"),   # Qwen2.5-14B MLP
    (64, 7, "bf16"),         # odd nf: the last unit is one row per block
    (1000, 130, "f32"),      # 4000-byte f32 rows
    (4096, 1, "bf16"),       # a single unit of one row pair
    (8, 5, "bf16"),          # 16-byte rows
    (2048, 3001, "f32"),     # 8 KB f32 rows: one CTA per SM, ragged last unit
]


def factors(orc, W, x, nf):
    """The oracle's factors of each output: silu(gate_i) and up_i (double), for the floor of the
    product rule."""
    y = orc.matvec(W, x)
    return np.array([orc.silu(v) for v in y[:nf]]), y[nf:]


def ffn_inputs(H, nf, wdt, layer):
    W = synth.ffn_weight_rows(SEED, layer, 0, 2 * nf, H, wdt)
    x = synth.hidden(SEED, 100 + layer, 0, H)
    return W, x


def run_step(qkv, H, nf, wdt, W, x):
    import torch
    dW, dx = to_dev(W), to_dev(x)
    out = torch.full((nf,), float("nan"), dtype=torch.float32, device="cuda")
    dt = qkv.QKV_BF16 if wdt == "bf16" else qkv.QKV_F32
    qkv.qkv_ffn_step(H, nf, dt, dx, dW, out, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    flags, _ = qkv.qkv_check_device_error()
    assert flags == 0
    return to_host(out)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "H%d_nf%d_%s" % s)
def test_ffn_matches_oracle(orc, qkv, shape):
    H, nf, wdt = shape
    W, x = ffn_inputs(H, nf, wdt, layer=2)
    got = run_step(qkv, H, nf, wdt, W, x)
    want = orc.ffn_swiglu(W, x)
    assert_product_close(got, want, *factors(orc, W, x, nf), "ffn %s" % (shape,))


def test_ffn_graph_equals_steps_bitwise(qkv):
    """Three layers of one shape: graph replay (twice) == three qkv_ffn_step calls."""
    import torch
    H, nf, wdt = 5120, 1536, "bf16"
    dt = qkv.QKV_BF16
    layers, outs_graph, outs_step = [], [], []
    for layer in range(3):
        W, x = ffn_inputs(H, nf, wdt, layer=10 + layer)
        dW, dx = to_dev(W), to_dev(x)
        og = torch.full((nf,), float("nan"), dtype=torch.float32, device="cuda")
        os_ = torch.full((nf,), float("nan"), dtype=torch.float32, device="cuda")
        layers.append(dict(x=dx, w_gate_up=dW, out=og))
        outs_graph.append(og)
        outs_step.append((dx, dW, os_))
    stream = torch.cuda.Stream()
    g = qkv.qkv_ffn_graph_create(H, nf, dt, layers, stream)
    assert g.kernel_count == 3
    for _ in range(2):
        g.launch(stream)
    stream.synchronize()
    for dx, dW, os_ in outs_step:
        qkv.qkv_ffn_step(H, nf, dt, dx, dW, os_, stream=stream.cuda_stream)
    stream.synchronize()
    for og, (_, _, os_) in zip(outs_graph, outs_step):
        a, b = to_host(og), to_host(os_)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("w", [configs.QWEN05_FFN, configs.QWEN7B_FFN, configs.QWEN14B_FFN], ids=lambda w: w.name)
def test_ffn_model_graph_full_size(orc, qkv, w):
    """The L-layer graph with the bench's inputs (seed 0, x of layer l = hidden(100 + l)):
    every layer's output against the oracle, and the first and last layers against a
    direct qkv_ffn_step, bitwise."""
    import torch
    L = w.n_layers
    dt = qkv.QKV_BF16 if w.w_dtype == "bf16" else qkv.QKV_F32
    dx = torch.empty(L, w.hidden, dtype=torch.float32, device="cuda")
    dout = torch.full((L, w.n_ff), float("nan"), dtype=torch.float32, device="cuda")
    hostW = np.empty((2 * w.n_ff, w.hidden), np.uint16 if w.w_dtype == "bf16" else np.float32)
    layers, keep, want = [], [], []
    for l in range(L):
        synth.ffn_weight_rows(SEED, l, 0, 2 * w.n_ff, w.hidden, w.w_dtype, out=hostW)
        x = synth.hidden(SEED, 100 + l, 0, w.hidden)
        want.append((orc.ffn_swiglu(hostW, x),) + factors(orc, hostW, x, w.n_ff))
        dW = to_dev(hostW)
        dx[l].copy_(to_dev(x))
        keep.append(dW)
        layers.append(dict(x=dx[l], w_gate_up=dW, out=dout[l]))
    stream = torch.cuda.Stream()
    g = qkv.qkv_ffn_graph_create(w.hidden, w.n_ff, dt, layers, stream)
    assert g.kernel_count == L
    torch.cuda.synchronize()
    g.launch(stream)
    stream.synchronize()
    flags, _ = qkv.qkv_check_device_error(stream)
    assert flags == 0
    got = to_host(dout)
    for l in range(L):
        assert_product_close(got[l], *want[l], "%s layer %d" % (w.name, l))
    for l in (0, L - 1):
        o = torch.full((w.n_ff,), float("nan"), dtype=torch.float32, device="cuda")
        qkv.qkv_ffn_step(w.hidden, w.n_ff, dt, dx[l], keep[l], o, stream=stream.cuda_stream)
        stream.synchronize()
        assert np.array_equal(to_host(o).view(np.uint32), got[l].view(np.uint32))
