"""Whole-model decode steps captured in one CUDA graph, against the oracle.

  * Qwen2.5-0.5B shape, 24 layers, f32 weights, f16 cache of 2048 rows,
    128 decode steps at positions 0..127 (x of every layer re-seeded per
    step, copied in before each replay, position advanced on the device);
  * Qwen2.5-7B shape, 28 layers, bf16 weights, f16 cache, position 1641;
  * Qwen2.5-14B shape, 48 layers (0-23 concat, 24-47 mixed), position 3254;
  * the same 7B and 14B models with the RMSNorm prologue fused into every layer
    (the graph the normed workloads time), on hidden states of a different
    RMS per layer.
Every output and both cache regions of every layer are compared.  Replay is
also checked bit-for-bit against sequential decode calls, and the graph's
kernel count (launches per step) against one launch per layer.
"""
import numpy as np
import pytest

import qkv_rope_kv_gb300 as Q
from gpu_helpers import HostLayer, assert_f32_close, assert_kv_region, canary, to_dev, to_host
from qkv_rope_kv_gb300 import configs, synth

pytestmark = pytest.mark.gpu

DT = {"f32": Q.QKV_F32, "bf16": Q.QKV_BF16, "f16": Q.QKV_F16}


class DeviceModel:
    """Device buffers of an L-layer model: x block, output block, weights, caches."""

    def __init__(self, w: configs.Workload, seed=0, keep_host=True):
        import torch
        self.w = w
        self.layers = [HostLayer(w.hidden, w.n_head, w.n_head_kv, w.head_dim, w.w_dtype, l, seed)
                       for l in range(w.n_layers)] if keep_host else None
        self.plans = {}
        for cls in (Q.QKV_CLASS_CONCAT, Q.QKV_CLASS_MIXED):
            self.plans[cls] = Q.qkv_plan_create(w.hidden, w.n_head, w.n_head_kv, w.head_dim, w.theta,
                                                w.n_ctx, w_dtype=DT[w.w_dtype], kv_dtype=DT[w.kv_dtype],
                                                layer_class=cls)
        self.dx = torch.zeros(w.n_layers, w.hidden, dtype=torch.float32, device="cuda")
        self.dout = torch.zeros(w.n_layers, w.rows, dtype=torch.float32, device="cuda")
        self.dpos = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.dW, self.db, self.dk, self.dv = [], [], [], []
        self.kv0 = []
        for l, L in enumerate(self.layers):
            self.dW.append(to_dev(L.W))
            self.db.append(to_dev(L.bias))
            k0, v0 = canary(w.n_ctx, w.nkt, w.kv_dtype, 2 * l), canary(w.n_ctx, w.nkt, w.kv_dtype, 2 * l + 1)
            self.kv0.append((k0, v0))
            self.dk.append(to_dev(k0))
            self.dv.append(to_dev(v0))
        self.norms = [synth.norm_weight(seed, l, w.hidden) for l in range(w.n_layers)] if w.rmsnorm else None
        self.dnorm = [to_dev(n) for n in self.norms] if w.rmsnorm else None

    def h(self, l, pos):
        """The layer's input: x itself, or, for a normed model, a hidden state whose RMS
        differs per layer (0.25 .. 6) so that the fused normalisation matters."""
        x = self.layers[l].x(pos)
        if not self.w.rmsnorm:
            return x
        return (np.float32(2.0 ** (l % 5 - 2) * (1.0 + 0.25 * (l % 3))) * x).astype(np.float32)

    def cls(self, l):
        return Q.QKV_CLASS_MIXED if l in self.w.mixed_layers else Q.QKV_CLASS_CONCAT

    def layer_ptrs(self, l):
        w = self.w
        a, b = w.nqt, w.nqt + w.nkt
        o = self.dout[l]
        d = dict(x=self.dx[l], q=o[:a], k=o[a:b], v=o[b:], kv_k=self.dk[l], kv_v=self.dv[l])
        if self.cls(l) == Q.QKV_CLASS_CONCAT:
            d.update(w=self.dW[l], bias=self.db[l])
        else:
            W, bb = self.dW[l], self.db[l]
            d.update(wq=W[:a], wk=W[a:b], wv=W[b:], bias_q=bb[:a], bias_k=bb[a:b], bias_v=bb[b:])
        return d

    def graph(self, stream):
        if self.w.rmsnorm:
            return Q.qkv_model_graph_create_rmsnorm([self.plans[self.cls(l)] for l in range(self.w.n_layers)],
                                                    [self.layer_ptrs(l) for l in range(self.w.n_layers)],
                                                    self.dnorm, self.w.rms_eps, self.dpos, stream)
        return Q.qkv_model_graph_create([self.plans[self.cls(l)] for l in range(self.w.n_layers)],
                                        [self.layer_ptrs(l) for l in range(self.w.n_layers)],
                                        self.dpos, stream)

    def set_step(self, pos):
        import torch
        xs = np.stack([self.h(l, pos) for l in range(self.w.n_layers)])
        self.dx.copy_(torch.from_numpy(xs))
        self.dpos.fill_(pos)

    def sequential_step(self, stream):
        for l in range(self.w.n_layers):
            p = self.layer_ptrs(l)
            if self.cls(l) == Q.QKV_CLASS_CONCAT:
                Q.qkv_decode_step(self.plans[self.cls(l)], p["x"], p["w"], p["bias"], self.dpos, p["q"],
                                  p["k"], p["v"], p["kv_k"], p["kv_v"], stream)
            else:
                Q.qkv_decode_step_mixed(self.plans[self.cls(l)], p["x"], p["wq"], p["wk"], p["wv"],
                                        p["bias_q"], p["bias_k"], p["bias_v"], self.dpos, p["q"],
                                        p["k"], p["v"], p["kv_k"], p["kv_v"], stream)


def oracle_model_step(orc, model, pos, kv_state):
    """Oracle outputs [L, R] for one step; kv_state (list of (k, v)) is updated in place."""
    w = model.w
    outs = np.empty((w.n_layers, w.rows), np.float32)
    a, b = w.nqt, w.nqt + w.nkt
    for l, L in enumerate(model.layers):
        kk, vv = kv_state[l]
        x = model.h(l, pos)
        if w.rmsnorm:
            x = orc.rmsnorm(x, model.norms[l], w.rms_eps)
        if model.cls(l) == Q.QKV_CLASS_CONCAT:
            st, q, k, v = orc.decode(L.W, x, L.bias, w.n_head, w.n_head_kv, w.head_dim, w.theta,
                                     w.freq_scale, pos, kk, vv)
        else:
            Wq, Wk, Wv = L.sections()
            st, q, k, v = orc.decode_mixed(Wq, Wk, Wv, x, L.bias, w.n_head, w.n_head_kv, w.head_dim,
                                           w.theta, w.freq_scale, pos, kk, vv)
        assert st == 0
        outs[l] = np.concatenate([q, k, v])
    return outs


def check_outputs(model, got, want, what):
    w = model.w
    a, b = w.nqt, w.nqt + w.nkt
    for l in range(w.n_layers):
        assert_f32_close(got[l, :a], want[l, :a], "%s layer %d q" % (what, l))
        assert_f32_close(got[l, a:b], want[l, a:b], "%s layer %d k" % (what, l))
        assert_f32_close(got[l, b:], want[l, b:], "%s layer %d v" % (what, l))


def check_caches(model, kv_state, rows, want_outs_last):
    w = model.w
    kvt = np.float32 if w.kv_dtype == "f32" else np.uint16
    a, b = w.nqt, w.nqt + w.nkt
    for l in range(w.n_layers):
        assert_kv_region(to_host(model.dk[l], kvt), kv_state[l][0], rows, "layer %d K" % l,
                         section_f32=want_outs_last[l, a:b])
        assert_kv_region(to_host(model.dv[l], kvt), kv_state[l][1], rows, "layer %d V" % l,
                         section_f32=want_outs_last[l, b:])


def _single_step_model(orc, w):
    import torch
    model = DeviceModel(w)
    stream = torch.cuda.Stream()
    g = model.graph(stream)
    assert g.kernel_count == w.n_layers
    pos = w.positions[0]
    model.set_step(pos)
    torch.cuda.synchronize()
    g.launch(stream)
    stream.synchronize()
    kv_state = [(k.copy(), v.copy()) for k, v in model.kv0]
    want = oracle_model_step(orc, model, pos, kv_state)
    got = to_host(model.dout)
    check_outputs(model, got, want, w.name)
    check_caches(model, kv_state, [pos], want)
    assert Q.qkv_check_device_error(stream)[0] == 0
    return model, g, stream


def test_qwen7b_28_layers(orc, qkv):
    _single_step_model(orc, configs.QWEN7B)


def test_qwen14b_48_layers_mixed_classes(orc, qkv):
    import torch
    model, g, stream = _single_step_model(orc, configs.QWEN14B)
    # replay == sequential decode calls, bit for bit (fresh caches for both)
    first = to_host(model.dout).copy()
    caches = [(to_host(k).copy(), to_host(v).copy()) for k, v in zip(model.dk, model.dv)]
    for l in range(model.w.n_layers):
        model.dk[l].copy_(to_dev(model.kv0[l][0]))
        model.dv[l].copy_(to_dev(model.kv0[l][1]))
    model.dout.zero_()
    torch.cuda.synchronize()
    model.sequential_step(stream)
    stream.synchronize()
    assert np.array_equal(to_host(model.dout).view(np.uint32), first.view(np.uint32))
    for l in range(model.w.n_layers):
        assert np.array_equal(to_host(model.dk[l]), caches[l][0])
        assert np.array_equal(to_host(model.dv[l]), caches[l][1])


def test_qwen05_24_layer_sweep_128_steps(orc, qkv):
    import torch
    w = configs.QWEN05_SWEEP
    model = DeviceModel(w)
    stream = torch.cuda.Stream()
    g = model.graph(stream)
    assert g.kernel_count == w.n_layers
    kv_state = [(k.copy(), v.copy()) for k, v in model.kv0]
    want = None
    for pos in w.positions:
        with torch.cuda.stream(stream):
            model.set_step(pos)
        g.launch(stream)
        stream.synchronize()
        want = oracle_model_step(orc, model, pos, kv_state)
        check_outputs(model, to_host(model.dout), want, "%s pos %d" % (w.name, pos))
    check_caches(model, kv_state, list(w.positions), want)
    assert Q.qkv_check_device_error(stream)[0] == 0


def test_run_host_matches_device_replay(orc, qkv):
    """The host-buffer entry point (copy in, replay, copy out) gives the same bits."""
    import torch
    w = configs.Workload("small-host", 1024, 8, 2, 64, "bf16", "f16", 64, 3, (9,), mixed_layers=(1,))
    model = DeviceModel(w)
    stream = torch.cuda.Stream()
    g = model.graph(stream)
    xs = np.stack([L.x(9) for L in model.layers]).astype(np.float32)
    h_in = torch.from_numpy(xs).pin_memory()
    h_out = torch.empty(w.n_layers, w.rows, dtype=torch.float32).pin_memory()
    model.dpos.fill_(9)
    torch.cuda.synchronize()
    g.run_host(h_in, model.dx, model.dout, h_out, stream)
    stream.synchronize()
    kv_state = [(k.copy(), v.copy()) for k, v in model.kv0]
    want = oracle_model_step(orc, model, 9, kv_state)
    check_outputs(model, h_out.numpy(), want, "run_host")
    assert np.array_equal(h_out.numpy().view(np.uint32), to_host(model.dout).view(np.uint32))


def test_run_host_calls_in_a_row(orc, qkv):
    """Four run_host calls enqueued back to back (each with its own host input and output
    buffers, one synchronisation at the end): the input copy of a call overlaps the output
    copy of the one before, and every call's outputs are its own step's, against the
    oracle.  The position travels in the input block, as in the bench's host path."""
    import torch
    w = configs.Workload("small-host-seq", 1024, 8, 2, 64, "bf16", "f16", 64, 3, (9,), mixed_layers=(1,))
    model = DeviceModel(w)
    x_off = 256
    in_bytes = x_off + w.n_layers * w.hidden * 4
    block = torch.zeros(in_bytes, dtype=torch.uint8, device="cuda")
    model.dpos = block[:4].view(torch.int32)
    model.dx = block[x_off:].view(torch.float32).view(w.n_layers, w.hidden)
    stream = torch.cuda.Stream()
    g = model.graph(stream)
    positions = [3, 17, 40, 63]
    h_ins, h_outs = [], []
    for p in positions:
        h = torch.zeros(in_bytes, dtype=torch.uint8)
        h[:4].view(torch.int32)[0] = p
        h[x_off:].view(torch.float32).view(w.n_layers, w.hidden).copy_(
            torch.from_numpy(np.stack([L.x(p) for L in model.layers]).astype(np.float32)))
        h_ins.append(h.pin_memory())
        h_outs.append(torch.full((w.n_layers, w.rows), float("nan"), dtype=torch.float32).pin_memory())
    torch.cuda.synchronize()
    for h_in, h_out in zip(h_ins, h_outs):
        g.run_host(h_in, block, model.dout, h_out, stream)
    stream.synchronize()
    kv_state = [(k.copy(), v.copy()) for k, v in model.kv0]
    for p, h_out in zip(positions, h_outs):
        want = oracle_model_step(orc, model, p, kv_state)
        check_outputs(model, h_out.numpy(), want, "run_host pos %d" % p)
    check_caches(model, kv_state, positions, want)
    assert Q.qkv_check_device_error(stream)[0] == 0


def test_qwen7b_28_layers_rmsnorm(orc, qkv):
    _single_step_model(orc, configs.QWEN7B_NORM)


def test_qwen14b_48_layers_mixed_rmsnorm(orc, qkv):
    """Every layer of the normed 14B graph against the oracle, then the graph against
    sequential normed steps of its concat layers (the mixed class has no normed
    single-step entry point; its layers are covered by the oracle comparison)."""
    import torch
    w = configs.QWEN14B_NORM
    model, g, stream = _single_step_model(orc, w)
    first = to_host(model.dout).copy()
    a, b = w.nqt, w.nqt + w.nkt
    plan = model.plans[Q.QKV_CLASS_CONCAT]
    for l in range(0, w.n_layers, 7):
        if model.cls(l) != Q.QKV_CLASS_CONCAT:
            continue
        out = torch.empty(w.rows, dtype=torch.float32, device="cuda")
        dk, dv = to_dev(model.kv0[l][0]), to_dev(model.kv0[l][1])
        Q.qkv_decode_step_rmsnorm(plan, model.dx[l], model.dnorm[l], w.rms_eps, model.dW[l], model.db[l],
                                  model.dpos, out[:a], out[a:b], out[b:], dk, dv, stream=stream)
        stream.synchronize()
        assert np.array_equal(to_host(out).view(np.uint32), first[l].view(np.uint32)), "layer %d" % l
        assert torch.equal(dk, model.dk[l]) and torch.equal(dv, model.dv[l]), "layer %d cache" % l
