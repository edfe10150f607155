"""Benchmark of the decode attention-input stage on GB300.

Default workload: Qwen2.5-14B shape, 48 layers (0-23 concat class, 24-47
mixed class), bf16 weights, f16 KV cache of 4096 rows, decode at position
3254.  One step = one replay of the whole-model CUDA graph (48 fused
projection+epilogue launches).  Metric: decode QKV layers/s (whole job) and
achieved HBM GB/s of the projection kernel against the measured copy peak.

  python bench.py [--steps K] [--warmup W] [--impl native|reference] [--workload NAME]
  torchrun --nproc-per-node N bench.py --gpus N ...   (independent replicas per GPU)

Timing: CUDA events on the replay stream around K replays, barrier and
synchronise on both sides, max over ranks.  Every step reads 3.5 GB of
weights, far more than the 126 MB L2, so no flush is needed between steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from qkv_rope_kv_gb300 import configs  # noqa: E402
from qkv_rope_kv_gb300 import synth  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 1024 * 1024
METRIC = "decode QKV layers/sec and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=configs.QWEN14B.name,
                    choices=sorted(configs.WORKLOADS) + sorted(configs.FFN_WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="bound on the oracle's CPU-baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU-baseline leg")
    ap.add_argument("--no-workloads", action="store_true",
                    help="default workload only: skip timing the other configurations")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling captures only: run the first N layers of the workload "
                         "(the result is not a bench number and says so)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(rel_path: str) -> str:
    """SHA-256 of a kernel source with its comments and blank lines removed: a traffic
    capture stays valid across comment edits, and only across those."""
    import re
    with open(os.path.join(ROOT, rel_path), encoding="utf-8") as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def traffic_per_launch(workload_name: str):
    """(DRAM bytes per launch, kernel) of the workload's dominant kernel from a committed ncu
    capture, if that kernel's source file is unchanged since the capture; else (None, None)."""
    try:
        with open(TRAFFIC_FILE) as fh:
            t = json.load(fh)["captures"][workload_name]
        if t["source_sha256"] != source_hash(t["source"]):
            return None, None
        return int(t["bytes_per_launch"]), t["kernel"]
    except Exception:
        return None, None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s, p in zip(sm, pw) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------- device model

def build_model(w: configs.Workload, seed: int, sweep: bool = False):
    """Seeded weights, bias, inputs and zeroed caches for all layers, resident on the device.
    With ``sweep``, also one input block per decode position of the workload (position and the
    x of every layer seeded by (layer, position)), resident on the device."""
    import torch
    import qkv_rope_kv_gb300 as Q

    dt = {"f32": Q.QKV_F32, "bf16": Q.QKV_BF16, "f16": Q.QKV_F16}
    L = w.n_layers
    pos = w.positions[0]
    plans = {cls: Q.qkv_plan_create(w.hidden, w.n_head, w.n_head_kv, w.head_dim, w.theta, w.n_ctx,
                                    w_dtype=dt[w.w_dtype], kv_dtype=dt[w.kv_dtype], layer_class=cls,
                                    freq_scale=w.freq_scale)
             for cls in (Q.QKV_CLASS_CONCAT, Q.QKV_CLASS_MIXED)}
    # one input block per step: [position | pad | x of every layer], one output block [L, R]
    x_off = 256
    in_bytes = x_off + L * w.hidden * 4
    inbuf = torch.zeros(in_bytes, dtype=torch.uint8, device="cuda")
    dpos = inbuf[:4].view(torch.int32)
    dx = inbuf[x_off:].view(torch.float32).view(L, w.hidden)
    dout = torch.zeros(L, w.rows, dtype=torch.float32, device="cuda")
    wt = torch.int16 if w.w_dtype == "bf16" else torch.float32
    kvt = torch.int16 if w.kv_dtype == "f16" else torch.float32
    host_x = np.stack([synth.hidden(seed, l, pos, w.hidden) for l in range(L)])
    a, b = w.nqt, w.nqt + w.nkt
    layers, keep = [], []
    hostW = np.empty((w.rows, w.hidden), np.uint16 if w.w_dtype == "bf16" else np.float32)
    for l in range(L):
        synth.weight_rows(seed, l, 0, w.rows, w.hidden, w.w_dtype, out=hostW)
        dW = torch.from_numpy(hostW.view(np.int16) if w.w_dtype == "bf16" else hostW).to("cuda")
        db = torch.from_numpy(synth.bias(seed, l, w.rows)).to("cuda")
        dk = torch.zeros(w.n_ctx, w.nkt, dtype=kvt, device="cuda")
        dv = torch.zeros_like(dk)
        o = dout[l]
        d = dict(x=dx[l], q=o[:a], k=o[a:b], v=o[b:], kv_k=dk, kv_v=dv)
        if l in w.mixed_layers:
            d.update(wq=dW[:a], wk=dW[a:b], wv=dW[b:], bias_q=db[:a], bias_k=db[a:b], bias_v=db[b:])
        else:
            d.update(w=dW, bias=db)
        layers.append(d)
        keep += [dW, db, dk, dv]
    norms = [torch.from_numpy(synth.norm_weight(seed, l, w.hidden)).to("cuda") for l in range(L)] \
        if w.rmsnorm else None
    qk_norms = [tuple(torch.from_numpy(a).to("cuda") for a in synth.qk_norm_weights(seed, l, w.head_dim))
                for l in range(L)] if w.qknorm else None
    layer_plans = [plans[Q.QKV_CLASS_MIXED if l in w.mixed_layers else Q.QKV_CLASS_CONCAT] for l in range(L)]
    h_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    h_in[:4].view(torch.int32)[0] = pos
    h_in[x_off:].view(torch.float32).view(L, w.hidden).copy_(torch.from_numpy(host_x))
    inbuf.copy_(h_in)
    h_out = torch.empty(L, w.rows, dtype=torch.float32).pin_memory()
    blocks = None
    if sweep:
        # block i: [position i | pad | x of every layer at position i], the layout of inbuf
        hb = torch.zeros(len(w.positions), in_bytes, dtype=torch.uint8)
        for i, p_ in enumerate(w.positions):
            hb[i, :4].view(torch.int32)[0] = p_
            hb[i, x_off:].view(torch.float32).view(L, w.hidden).copy_(
                torch.from_numpy(np.stack([synth.hidden(seed, l, p_, w.hidden) for l in range(L)])))
        blocks = hb.to("cuda")
    torch.cuda.synchronize()
    return dict(plans=plans, layer_plans=layer_plans, layers=layers, norms=norms, qk_norms=qk_norms, keep=keep,
                inbuf=inbuf,
                dpos=dpos, dx=dx, dout=dout, h_in=h_in, h_out=h_out, in_bytes=in_bytes, blocks=blocks)


def time_replays(fn, steps: int, stream, flush=None):
    """Seconds of `steps` calls of fn on `stream`, timed with CUDA events on that stream.
    With `flush` (a device byte buffer larger than L2), the buffer is rewritten before
    every step, outside the timed events, so no step finds its weights in L2."""
    import torch
    if flush is None:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            fn()
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / 1e3
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i, (s0, s1) in enumerate(evs):
            flush.fill_(i & 0xFF)
            s0.record(stream)
            fn()
            s1.record(stream)
    stream.synchronize()
    return sum(s0.elapsed_time(s1) for s0, s1 in evs) / 1e3


def l2_flush_buffer(weight_bytes_per_step: int):
    """A 256 MB device buffer to flush L2 between steps when a step's weights would fit in
    (a few times) the 126 MB L2, else None."""
    import torch
    if weight_bytes_per_step > 4 * L2_BYTES:
        return None
    return torch.empty(256 << 20, dtype=torch.uint8, device="cuda")


def barrier_sync(world):
    import torch
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()


def max_over_ranks(v: float, world: int) -> float:
    from qkv_rope_kv_gb300 import shard
    return v if world == 1 else shard.max_over_ranks(v, device="cuda")


# ---------------------------------------------------------------- CPU baseline (oracle)

def oracle_layers_per_s(w: configs.Workload, seed: int, seconds: float, max_layers: int | None = None):
    """Time the oracle (single thread, as it stands) over consecutive layers of the workload
    until `seconds` of oracle time have been spent; weight generation is not timed."""
    import oracle
    orc = oracle.Oracle()
    pos = w.positions[0]
    done, spent = 0, 0.0
    kk = np.zeros((w.n_ctx, w.nkt), np.float32 if w.kv_dtype == "f32" else np.uint16)
    vv = kk.copy()
    a, b = w.nqt, w.nqt + w.nkt
    l = 0
    while (done == 0 or spent < seconds) and (max_layers is None or done < max_layers):
        layer = l % w.n_layers
        W = synth.weight_rows(seed, layer, 0, w.rows, w.hidden, w.w_dtype)
        bias = synth.bias(seed, layer, w.rows)
        x = synth.hidden(seed, layer, pos, w.hidden)
        nw = synth.norm_weight(seed, layer, w.hidden) if w.rmsnorm else None
        qkn = synth.qk_norm_weights(seed, layer, w.head_dim) if w.qknorm else None
        t0 = time.perf_counter()
        if nw is not None:
            x = orc.rmsnorm(x, nw, w.rms_eps)
        if qkn is not None:
            orc.decode_qknorm(W, x, bias, qkn[0], qkn[1], w.qk_eps, w.n_head, w.n_head_kv, w.head_dim, w.theta,
                              w.freq_scale, pos, kk, vv)
        elif layer in w.mixed_layers:
            orc.decode_mixed(W[:a], W[a:b], W[b:], x, bias, w.n_head, w.n_head_kv, w.head_dim,
                             w.theta, w.freq_scale, pos, kk, vv)
        else:
            orc.decode(W, x, bias, w.n_head, w.n_head_kv, w.head_dim, w.theta, w.freq_scale, pos, kk, vv)
        spent += time.perf_counter() - t0
        done += 1
        l += 1
    return done / spent, done, spent


# ---------------------------------------------------------------- oracle on all host cores

def _oracle_inputs(w, seed: int, layer: int):
    """Seeded inputs of one layer for the oracle (not timed)."""
    if isinstance(w, configs.FfnWorkload):
        return (synth.ffn_weight_rows(seed, layer, 0, 2 * w.n_ff, w.hidden, w.w_dtype),
                synth.hidden(seed, 100 + layer, 0, w.hidden))
    return (synth.weight_rows(seed, layer, 0, w.rows, w.hidden, w.w_dtype), synth.bias(seed, layer, w.rows),
            synth.hidden(seed, layer, w.positions[0], w.hidden),
            synth.norm_weight(seed, layer, w.hidden) if w.rmsnorm else None,
            synth.qk_norm_weights(seed, layer, w.head_dim) if w.qknorm else None)


def _oracle_run(orc, w, layer: int, inp, kv):
    if isinstance(w, configs.FfnWorkload):
        orc.ffn_swiglu(inp[0], inp[1])
        return
    W, bias, x, nw, qkn = inp
    if nw is not None:
        x = orc.rmsnorm(x, nw, w.rms_eps)
    kk, vv = kv
    a, b = w.nqt, w.nqt + w.nkt
    if qkn is not None:
        # the mixed class computes the same stage from three sections of the same rows
        orc.decode_qknorm(W, x, bias, qkn[0], qkn[1], w.qk_eps, w.n_head, w.n_head_kv, w.head_dim, w.theta,
                          w.freq_scale, w.positions[0], kk, vv)
    elif layer in w.mixed_layers:
        orc.decode_mixed(W[:a], W[a:b], W[b:], x, bias, w.n_head, w.n_head_kv, w.head_dim, w.theta,
                         w.freq_scale, w.positions[0], kk, vv)
    else:
        orc.decode(W, x, bias, w.n_head, w.n_head_kv, w.head_dim, w.theta, w.freq_scale, w.positions[0], kk, vv)


def _oracle_worker(w, seed: int, layers, start, stop, results):
    """One host process: generate its layers' inputs, then per round wait for the start
    barrier and run the oracle once per layer, reporting the oracle time; a round that
    starts with `stop` set ends the process."""
    sys.path.insert(0, ROOT)
    import oracle
    orc = oracle.Oracle()
    inputs = [_oracle_inputs(w, seed, l) for l in layers]
    kv = None
    if not isinstance(w, configs.FfnWorkload):
        kk = np.zeros((w.n_ctx, w.nkt), np.float32 if w.kv_dtype == "f32" else np.uint16)
        kv = (kk, kk.copy())
    while True:
        start.wait()
        if stop.value:
            return
        t0 = time.perf_counter()
        for l, inp in zip(layers, inputs):
            _oracle_run(orc, w, l, inp, kv)
        results.put(time.perf_counter() - t0)


def oracle_all_cores(w, seed: int, seconds: float = 0.0, rounds: int | None = None, warmup: int = 0):
    """Run the unmodified oracle in one spawned process per host core, all at once, one
    layer each per round (a round is timed by its slowest process).  Runs `rounds` rounds,
    or until about `seconds` of CPU time, after `warmup` untimed rounds.  Returns
    (layers/s, cores, layers, seconds).  Spawned, not forked: the parent may hold a CUDA
    context."""
    import multiprocessing as mp
    import oracle
    oracle.load()  # build once here, not in every worker
    cores = len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    start = ctx.Barrier(cores + 1)
    stop = ctx.Value("b", 0)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w, seed, [i % w.n_layers], start, stop, results),
                         daemon=True)
             for i in range(cores)]
    for pr in procs:
        pr.start()
    total, done, r = 0.0, 0, 0
    try:
        while True:
            start.wait(timeout=180)
            t = max(results.get(timeout=300) for _ in range(cores))
            r += 1
            if r > warmup:
                total += t
                done += 1
            if (rounds is not None and done >= rounds) or (rounds is None and total * cores >= seconds):
                break
        stop.value = 1
        start.wait(timeout=60)
    finally:
        for pr in procs:
            pr.join(timeout=30)
            if pr.is_alive():
                pr.terminate()
    return cores * done / total, cores, cores * done, total


def cpu_baseline_leg(w, seed: int, seconds: float, what: str):
    """cpu_baseline: the oracle on all host cores, with the single-thread figure beside it."""
    v1, n1, s1 = (ffn_oracle_layers_per_s if isinstance(w, configs.FfnWorkload) else oracle_layers_per_s)(
        w, seed, seconds / 4, max_layers=w.n_layers)
    single = {"value": v1, "unit": "layers/s", "cores": 1,
              "sample": "%d consecutive layers (%.1f s), one thread" % (n1, s1)}
    try:
        v, cores, layers, secs = oracle_all_cores(w, seed, seconds=seconds)
    except Exception as exc:  # the pool is a baseline, never a reason to lose the GPU line
        return dict(single, kind="oracle", note="all-core run failed: %s" % str(exc)[:120])
    return {"value": v, "unit": "layers/s", "cores": cores, "kind": "oracle",
            "sample": "%s: one layer per process on %d processes at once (one per host core), %d layers in "
                      "%.2f s of wall time, about %.0f s of CPU; the C oracle as it stands (double "
                      "accumulation), input generation excluded" % (what, cores, layers, secs, secs * cores),
            "single_thread": single}


def reference_arm(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    # K timed steps after W untimed ones; a step is one oracle layer on every host core at once
    value, cores, layers, secs = oracle_all_cores(w, 0, rounds=args.steps, warmup=args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "layers/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64/Box-Muller weights, bias, x)",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "layers/s", "cores": cores, "kind": "oracle",
                         "sample": "%d steps x %d layers of %s at pos %d (one per process, one process per "
                                   "host core, at once), the C oracle as it stands (double accumulation), "
                                   "input generation excluded" % (args.steps, cores, w.name, w.positions[0])},
        "e2e": {"value": value, "unit": "layers/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w: configs.Workload):
    return {"workload": w.name, "layers": w.n_layers, "hidden": w.hidden,
            "heads": "%d/%d" % (w.n_head, w.n_head_kv), "head_dim": w.head_dim,
            "w_dtype": w.w_dtype, "kv_dtype": w.kv_dtype, "n_ctx": w.n_ctx, "pos": w.positions[0],
            "mixed_layers": "%d-%d" % (w.mixed_layers[0], w.mixed_layers[-1]) if w.mixed_layers else "none",
            "rmsnorm": ("fused in front of each projection, eps %g" % w.rms_eps) if w.rmsnorm else "none (x given)",
            "qk_norm": ("per-head q/k RMSNorm before RoPE (FusedQkvNorm), weights of %d values, eps %g"
                        % (w.head_dim, w.qk_eps)) if w.qknorm else "none",
            "l2": ("inputs larger than L2: %.2f GB of weights per step" % (w.n_layers * w.w_bytes() / 1e9))
            if w.n_layers * w.w_bytes() > 4 * L2_BYTES
            else "L2 flushed before every timed step (256 MB written outside the timed events); "
                 "%.1f MB of weights per step" % (w.n_layers * w.w_bytes() / 1e6),
            "parallelism": "replicas"}


# ---------------------------------------------------------------- native arm

def model_graph(m, w, stream):
    """The whole-model decode graph of a built model (plain, RMSNorm-fused or FusedQkvNorm)."""
    import torch
    import qkv_rope_kv_gb300 as Q
    if w.qknorm:
        plan0 = m["layer_plans"][0]
        m["qk_ws"] = torch.zeros(Q.qkv_qknorm_workspace_bytes(plan0) // 4, dtype=torch.int32, device="cuda")
        return Q.qkv_model_graph_create_qknorm(m["layer_plans"], m["layers"], [a for a, _ in m["qk_norms"]],
                                               [b for _, b in m["qk_norms"]], w.qk_eps, m["dpos"], m["qk_ws"],
                                               stream)
    if w.rmsnorm:
        return Q.qkv_model_graph_create_rmsnorm(m["layer_plans"], m["layers"], m["norms"], w.rms_eps, m["dpos"],
                                                stream)
    return Q.qkv_model_graph_create(m["layer_plans"], m["layers"], m["dpos"], stream)


def direct_step(m, w, stream):
    """For a one-layer decode workload without a fused norm, the step as a user makes it: one
    qkv_decode_step (or qkv_decode_step_mixed) launch, which starts on the device about 0.8 us
    sooner than a one-node graph; else None (the workload replays its model graph)."""
    import qkv_rope_kv_gb300 as Q
    if w.n_layers != 1 or w.rmsnorm or w.qknorm or len(w.positions) > 1:
        return None
    d, plan = m["layers"][0], m["layer_plans"][0]
    if "w" in d:
        return lambda: Q.qkv_decode_step(plan, d["x"], d["w"], d["bias"], m["dpos"], d["q"], d["k"], d["v"],
                                         d["kv_k"], d["kv_v"], stream)
    return lambda: Q.qkv_decode_step_mixed(plan, d["x"], d["wq"], d["wk"], d["wv"], d["bias_q"], d["bias_k"],
                                           d["bias_v"], m["dpos"], d["q"], d["k"], d["v"], d["kv_k"], d["kv_v"],
                                           stream)


def check_flags(stream, what: str):
    import qkv_rope_kv_gb300 as Q
    stream.synchronize()
    flags, _ = Q.qkv_check_device_error(stream)
    if flags:
        raise RuntimeError("device status flags set during %s: %#x" % (what, flags))


def roofline_entry(w, layers_per_step: int, elapsed: float, steps: int, launches: int, algo: int):
    """Throughput fields of one workload entry: layers/s, GB/s and the fractions of the peaks."""
    peak, peak_kind = measured_peak()
    per_layer = elapsed / steps / layers_per_step
    gbs = algo / per_layer / 1e9
    traffic, kernel = traffic_per_launch(w.name)
    return {"workload": w.name, "layers": layers_per_step, "steps": steps, "ms_per_step": 1e3 * elapsed / steps,
            "layers_per_s": layers_per_step * steps / elapsed, "hbm_gbs": gbs, "frac": gbs / peak,
            "peak": peak, "peak_kind": peak_kind, "frac_of_nominal_8000": gbs / NOMINAL_HBM_GBS,
            "algo_bytes_per_launch": algo, "traffic": traffic, "traffic_kernel": kernel,
            "launches_per_step": launches}


def decode_workload_entry(w, seed: int, steps: int):
    """One decode workload timed in this process: its whole-model graph replayed `steps` times
    (L2 flushed before every step when its weights would stay in L2).  A workload with several
    positions is a sweep: each step first copies that step's input block (position and the x of
    every layer, resident on the device) into the graph's input block, inside the timed region,
    so consecutive steps run consecutive positions."""
    import torch
    sweep = len(w.positions) > 1
    m = build_model(w, seed, sweep=sweep)
    stream = torch.cuda.Stream()
    graph = model_graph(m, w, stream)
    if sweep:
        blocks, inbuf, P = m["blocks"], m["inbuf"], len(w.positions)
        step_no = [0]

        def step():
            with torch.cuda.stream(stream):
                inbuf.copy_(blocks[step_no[0] % P], non_blocking=True)
            graph.launch(stream)
            step_no[0] += 1
    else:
        def step():
            graph.launch(stream)
    direct = direct_step(m, w, stream)
    if direct is not None:
        step = direct
    for _ in range(3):
        step()
    check_flags(stream, "warm-up of %s" % w.name)
    flush = l2_flush_buffer(w.n_layers * w.w_bytes())
    if sweep:
        step_no[0] = 0
    elapsed = time_replays(step, steps, stream, flush)
    check_flags(stream, w.name)
    e = roofline_entry(w, w.n_layers, elapsed, steps, graph.kernel_count, w.algo_bytes_per_layer())
    e["config"] = workload_config(w)
    if direct is not None:
        e["step"] = "one qkv_decode_step launch per step (no graph)"
    if sweep:
        e["sweep"] = ("positions %d..%d in order, one per step (%d sweeps); each step copies its %d-byte input "
                      "block (position + x of every layer, device resident) into the graph's input block inside "
                      "the timed region, then replays the %d-launch graph"
                      % (w.positions[0], w.positions[-1], steps // len(w.positions), m["in_bytes"], w.n_layers))
    del graph, m
    torch.cuda.synchronize()
    return e


def prefill_workload_entry(w, seed: int, steps: int, weights=None):
    """The prefill graph of workload w timed in this process.  `weights`, a list of (W, bias)
    device tensors per layer, reuses weights already on the device (the 14B decode model's
    concat weights are the prefill workload's, row for row)."""
    import torch
    model = build_prefill(w, seed, weights)
    stream = torch.cuda.Stream()
    graph = model["graph_fn"](stream)
    for _ in range(3):
        graph.launch(stream)
    check_flags(stream, "warm-up of %s" % w.name)
    elapsed = time_replays(lambda: graph.launch(stream), steps, stream)
    check_flags(stream, w.name)
    algo_b, algo_f = prefill_algo(w)
    e = roofline_entry(w, w.n_layers, elapsed, steps, graph.kernel_count, algo_b)
    e["tflops"] = algo_f / (elapsed / steps / w.n_layers) / 1e12
    e["algo_flops_per_launch"] = algo_f
    e["config"] = dict(workload_config(w), nt=w.nt, positions="0..%d" % (w.nt - 1))
    del graph, model
    torch.cuda.synchronize()
    return e


def workloads_leg(args, main_entry, main_model):
    """Every other configuration of the metric, timed in this process after the headline:
    7B 28 layers, 0.5B single layer (L2 flushed), 0.5B 24-layer sweep over positions 0..127,
    14B prefill of 128 tokens (on the headline model's weights)."""
    import torch
    out = {configs.QWEN14B.name: main_entry}
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t0 = time.time()
    plan = [(configs.QWEN7B, max(args.steps, 200)), (configs.QWEN05_SINGLE, max(args.steps, 500)),
            (configs.QWEN05_SWEEP, 2 * len(configs.QWEN05_SWEEP.positions))]
    for w, steps in plan:
        out[w.name] = decode_workload_entry(w, 0, steps)
    weights = [(main_model["keep"][4 * l], main_model["keep"][4 * l + 1]) for l in range(configs.QWEN14B.n_layers)]
    out[configs.QWEN14B_PREFILL.name] = prefill_workload_entry(configs.QWEN14B_PREFILL, 0, max(args.steps, 20),
                                                               weights)
    clk = clocks.stop()
    out["clocks"] = clk
    out["wall_s"] = time.time() - t0
    return out


def native_arm(args, w):
    import torch
    import qkv_rope_kv_gb300 as Q

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    Q.load()
    seed = rank  # each replica runs its own seeded model
    m = build_model(w, seed)
    stream = torch.cuda.Stream()
    graph = model_graph(m, w, stream)
    kernels = graph.kernel_count
    step = direct_step(m, w, stream) or (lambda: graph.launch(stream))

    for _ in range(max(args.warmup, 3)):
        step()
    stream.synchronize()
    flags, _ = Q.qkv_check_device_error(stream)
    if flags:
        raise RuntimeError("device status flags set during warm-up: %#x" % flags)

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier_sync(world)
    flush = l2_flush_buffer(w.n_layers * w.w_bytes())
    elapsed = time_replays(step, args.steps, stream, flush)
    barrier_sync(world)
    clk = clocks.stop()
    elapsed = max_over_ranks(elapsed, world)

    e2e = None
    if not args.no_e2e:
        h_in, h_out = m["h_in"], m["h_out"]
        for _ in range(3):
            graph.run_host(h_in, m["inbuf"], m["dout"], h_out, stream)
        barrier_sync(world)
        e_el = time_replays(lambda: graph.run_host(h_in, m["inbuf"], m["dout"], h_out, stream),
                            args.steps, stream, flush)
        barrier_sync(world)
        e_el = max_over_ranks(e_el, world)
        e2e = {"value": world * w.n_layers * args.steps / e_el, "unit": "layers/s",
               "h2d_bytes_per_step": int(m["in_bytes"]),
               "d2h_bytes_per_step": int(h_out.numel() * 4),
               "ms_per_step": 1e3 * e_el / args.steps,
               "path": "qkv_model_graph_run_host: pinned host x block + position -> device, "
                       "graph replay, q|k|v of all layers -> pinned host"}

    ms = 1e3 * elapsed / args.steps
    layers_per_s = world * w.n_layers * args.steps / elapsed
    per_layer_s = elapsed / args.steps / w.n_layers
    algo = w.algo_bytes_per_layer()
    achieved = algo / per_layer_s / 1e9
    peak, peak_kind = measured_peak()
    traffic, traffic_kernel = traffic_per_launch(w.name)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_leg(w, seed, args.cpu_seconds, "%s at pos %d" % (w.name, w.positions[0]))

    workloads = None
    if world == 1 and w.name == configs.QWEN14B.name and not args.no_workloads:
        main_entry = roofline_entry(w, w.n_layers, elapsed, args.steps, kernels, algo)
        main_entry["config"] = workload_config(w)
        main_entry["note"] = "the headline line's own measurement"
        del graph
        workloads = workloads_leg(args, main_entry, m)

    if rank == 0:
        line = {
            "metric": METRIC, "value": layers_per_s, "unit": "layers/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64/Box-Muller weights ~N(0,0.02), bias ~N(0,0.1), "
                    "x ~N(0,1); bf16 weights widened exactly, f32 accumulate)",
            "config": workload_config(w),
            "hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS,
                         "traffic": traffic, "algo_bytes_per_launch": algo,
                         "kernel": traffic_kernel or "qkv_decode ring kernel (fused projection + "
                                                     "bias/RoPE/KV-store tail)",
                         "duration_basis": "step time / %d launches (back-to-back graph replay)" % w.n_layers},
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": kernels * args.steps,
            "launches_per_step": kernels, "clocks": clk,
        }
        if workloads is not None:
            line["workloads"] = workloads
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def prefill_algo(w: configs.Workload):
    """Bytes and flops one prefill layer must move/do: W, X, bias read; Y and nt cache rows written."""
    bytes_ = (w.w_bytes() + w.nt * w.hidden * 2 + 4 * w.rows + 4 * w.nt * w.rows
              + 2 * w.nt * w.nkt * w.kv_elem_bytes())
    flops = 2 * w.nt * w.rows * w.hidden
    return bytes_, flops


def build_prefill(w, seed: int, weights=None):
    """Seeded prefill inputs of every layer on the device (X of nt tokens, positions 0..nt-1,
    zeroed caches, Y) and a function that captures the prefill graph on a stream.  `weights`:
    per-layer (W, bias) device tensors to reuse, else generated from the same seeds."""
    import torch
    import qkv_rope_kv_gb300 as Q
    plan = Q.qkv_plan_create(w.hidden, w.n_head, w.n_head_kv, w.head_dim, w.theta, w.n_ctx,
                             w_dtype=Q.QKV_BF16, kv_dtype=Q.QKV_F16 if w.kv_dtype == "f16" else Q.QKV_F32,
                             freq_scale=w.freq_scale)
    positions = torch.arange(w.nt, dtype=torch.int32, device="cuda")
    kvt = torch.int16 if w.kv_dtype == "f16" else torch.float32
    layers = []
    hostW = np.empty((w.rows, w.hidden), np.uint16)
    for l in range(w.n_layers):
        if weights is None:
            synth.weight_rows(seed, l, 0, w.rows, w.hidden, "bf16", out=hostW)
            dW = torch.from_numpy(hostW.view(np.int16)).to("cuda")
            db = torch.from_numpy(synth.bias(seed, l, w.rows)).to("cuda")
        else:
            dW, db = weights[l]
            assert tuple(dW.shape) == (w.rows, w.hidden) and dW.element_size() == 2
        layers.append(dict(
            X=torch.from_numpy(synth.prefill_x(seed, l, w.nt, w.hidden).view(np.int16)).to("cuda"),
            w=dW, bias=db, positions=positions,
            Y=torch.empty(w.nt, w.rows, dtype=torch.float32, device="cuda"),
            kv_k=torch.zeros(w.n_ctx, w.nkt, dtype=kvt, device="cuda"),
            kv_v=torch.zeros(w.n_ctx, w.nkt, dtype=kvt, device="cuda")))
    torch.cuda.synchronize()
    return {"plan": plan, "layers": layers,
            "graph_fn": lambda stream: Q.qkv_prefill_graph_create([plan] * w.n_layers, layers, w.nt, stream)}


def prefill_arm(args, w):
    import torch
    import qkv_rope_kv_gb300 as Q

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    Q.load()
    seed = rank
    stream = torch.cuda.Stream()
    graph = build_prefill(w, seed)["graph_fn"](stream)
    for _ in range(max(args.warmup, 3)):
        graph.launch(stream)
    stream.synchronize()
    flags, _ = Q.qkv_check_device_error(stream)
    if flags:
        raise RuntimeError("device status flags set during warm-up: %#x" % flags)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier_sync(world)
    elapsed = time_replays(lambda: graph.launch(stream), args.steps, stream)
    barrier_sync(world)
    clk = clocks.stop()
    elapsed = max_over_ranks(elapsed, world)
    per_layer = elapsed / args.steps / w.n_layers
    algo_b, algo_f = prefill_algo(w)
    peak, peak_kind = measured_peak()
    if rank == 0:
        line = {
            "metric": METRIC, "value": world * w.n_layers * args.steps / elapsed, "unit": "layers/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 x bf16 -> f32",
            "data": "synthetic (seeded SplitMix64/Box-Muller X ~N(0,1), W ~N(0,0.02), bias ~N(0,0.1))",
            "config": dict(workload_config(w), nt=w.nt, positions="0..%d" % (w.nt - 1)),
            "hbm_gbs": algo_b / per_layer / 1e9, "tflops": algo_f / per_layer / 1e12,
            "roofline": {"bound": "hbm", "achieved": algo_b / per_layer / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": algo_b / per_layer / 1e9 / peak, "peak_kind": peak_kind,
                         "frac_of_nominal_8000": algo_b / per_layer / 1e9 / NOMINAL_HBM_GBS,
                         "traffic": traffic_per_launch(w.name)[0], "algo_bytes_per_launch": algo_b,
                         "algo_flops_per_launch": algo_f,
                         "kernel": "qkv_prefill_kernel (tcgen05 bf16 GEMM + bias/RoPE/KV-store epilogue)",
                         "duration_basis": "step time / %d launches" % w.n_layers},
            "gpu_launches": graph.kernel_count * args.steps, "launches_per_step": graph.kernel_count,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- FusedFFN workloads

FFN_METRIC = "decode FusedFFN (gate|up GEMV + SwiGLU) layers/sec and achieved HBM GB/s, 1 GPU"


def ffn_config(w):
    return {"workload": w.name, "layers": w.n_layers, "hidden": w.hidden, "n_ff": w.n_ff,
            "w_dtype": w.w_dtype,
            "l2": ("inputs larger than L2: %.2f GB of weights per step" % (w.n_layers * w.w_bytes() / 1e9))
            if w.n_layers * w.w_bytes() > 4 * L2_BYTES
            else "L2 flushed before every timed step (256 MB written outside the timed events); "
                 "%.1f MB of weights per step" % (w.n_layers * w.w_bytes() / 1e6),
            "parallelism": "replicas"}


def ffn_arm(args, w):
    import torch
    import qkv_rope_kv_gb300 as Q

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    Q.load()
    seed = rank
    L = w.n_layers
    dt = Q.QKV_BF16 if w.w_dtype == "bf16" else Q.QKV_F32
    dx = torch.empty(L, w.hidden, dtype=torch.float32, device="cuda")
    dout = torch.zeros(L, w.n_ff, dtype=torch.float32, device="cuda")
    hostW = np.empty((2 * w.n_ff, w.hidden), np.uint16 if w.w_dtype == "bf16" else np.float32)
    layers, keep = [], []
    for l in range(L):
        synth.ffn_weight_rows(seed, l, 0, 2 * w.n_ff, w.hidden, w.w_dtype, out=hostW)
        dW = torch.from_numpy(hostW.view(np.int16) if w.w_dtype == "bf16" else hostW).to("cuda")
        keep.append(dW)
        layers.append(dict(x=dx[l], w_gate_up=dW, out=dout[l]))
    h_in = torch.from_numpy(np.stack([synth.hidden(seed, 100 + l, 0, w.hidden) for l in range(L)])).pin_memory()
    dx.copy_(h_in)
    h_out = torch.empty(L, w.n_ff, dtype=torch.float32).pin_memory()
    stream = torch.cuda.Stream()
    graph = Q.qkv_ffn_graph_create(w.hidden, w.n_ff, dt, layers, stream)
    for _ in range(max(args.warmup, 3)):
        graph.launch(stream)
    stream.synchronize()
    flags, _ = Q.qkv_check_device_error(stream)
    if flags:
        raise RuntimeError("device status flags set during warm-up: %#x" % flags)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier_sync(world)
    flush = l2_flush_buffer(L * w.w_bytes())
    elapsed = time_replays(lambda: graph.launch(stream), args.steps, stream, flush)
    barrier_sync(world)
    clk = clocks.stop()
    elapsed = max_over_ranks(elapsed, world)
    e2e = None
    if not args.no_e2e:
        for _ in range(3):
            graph.run_host(h_in, dx, dout, h_out, stream)
        barrier_sync(world)
        e_el = time_replays(lambda: graph.run_host(h_in, dx, dout, h_out, stream), args.steps, stream, flush)
        barrier_sync(world)
        e_el = max_over_ranks(e_el, world)
        e2e = {"value": world * L * args.steps / e_el, "unit": "layers/s",
               "h2d_bytes_per_step": int(h_in.numel() * 4), "d2h_bytes_per_step": int(h_out.numel() * 4),
               "ms_per_step": 1e3 * e_el / args.steps,
               "path": "qkv_model_graph_run_host: pinned host x block -> device, graph replay, "
                       "SwiGLU outputs of all layers -> pinned host"}
    per_layer = elapsed / args.steps / L
    algo = w.algo_bytes_per_layer()
    peak, peak_kind = measured_peak()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline_leg(w, seed, args.cpu_seconds, w.name)
    if rank == 0:
        line = {
            "metric": FFN_METRIC, "value": world * L * args.steps / elapsed, "unit": "layers/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded SplitMix64/Box-Muller weights ~N(0,0.02), x ~N(0,1); "
                    "bf16 weights widened exactly, f32 accumulate)",
            "config": ffn_config(w),
            "hbm_gbs": algo / per_layer / 1e9,
            "roofline": {"bound": "hbm", "achieved": algo / per_layer / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": algo / per_layer / 1e9 / peak, "peak_kind": peak_kind,
                         "frac_of_nominal_8000": algo / per_layer / 1e9 / NOMINAL_HBM_GBS,
                         "traffic": traffic_per_launch(w.name)[0], "algo_bytes_per_launch": algo,
                         "kernel": "qkv_decode_blk_kernel (gate|up GEMV + SwiGLU tail)",
                         "duration_basis": "step time / %d launches (back-to-back graph replay)" % L},
            "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": graph.kernel_count * args.steps, "launches_per_step": graph.kernel_count,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def ffn_oracle_layers_per_s(w, seed: int, seconds: float, max_layers: int | None = None):
    """Time the FusedFFN oracle (single thread, as it stands) over consecutive layers."""
    import oracle
    orc = oracle.Oracle()
    done, spent, l = 0, 0.0, 0
    while (done == 0 or spent < seconds) and (max_layers is None or done < max_layers):
        layer = l % w.n_layers
        W = synth.ffn_weight_rows(seed, layer, 0, 2 * w.n_ff, w.hidden, w.w_dtype)
        x = synth.hidden(seed, 100 + layer, 0, w.hidden)
        t0 = time.perf_counter()
        orc.ffn_swiglu(W, x)
        spent += time.perf_counter() - t0
        done += 1
        l += 1
    return done / spent, done, spent


def ffn_reference_arm(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    value, cores, layers, secs = oracle_all_cores(w, 0, rounds=args.steps, warmup=args.warmup)
    line = {
        "impl": "reference", "metric": FFN_METRIC, "value": value, "unit": "layers/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64/Box-Muller weights and x)",
        "config": ffn_config(w),
        "cpu_baseline": {"value": value, "unit": "layers/s", "cores": cores, "kind": "oracle",
                         "sample": "%d steps x %d layers of %s (one per process, one process per host core, "
                                   "at once), the C oracle as it stands (double accumulation), input "
                                   "generation excluded" % (args.steps, cores, w.name)},
        "e2e": {"value": value, "unit": "layers/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.workload in configs.FFN_WORKLOADS:
        import dataclasses
        w = configs.FFN_WORKLOADS[args.workload]
        if args.layers is not None:
            w = dataclasses.replace(w, name=w.name + "-first%d-layers-profiling-only" % args.layers,
                                    n_layers=args.layers)
        if args.impl == "reference":
            ffn_reference_arm(args, w)
        else:
            ffn_arm(args, w)
        return
    w = configs.WORKLOADS[args.workload]
    if args.layers is not None:
        import dataclasses
        w = dataclasses.replace(w, name=w.name + "-first%d-layers-profiling-only" % args.layers,
                                n_layers=args.layers,
                                mixed_layers=tuple(l for l in w.mixed_layers if l < args.layers))
    if args.impl == "reference":
        reference_arm(args, w)
    elif w.nt > 1:
        prefill_arm(args, w)
    else:
        native_arm(args, w)


if __name__ == "__main__":
    main()
