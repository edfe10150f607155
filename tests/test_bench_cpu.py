"""The benchmark's reference arm (the CPU oracle on host cores) runs without a GPU
and prints the contract's JSON line."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--workload", "qwen2.5-7b-28layer"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "layers/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))  # one oracle process per host core
    assert d["e2e"] == {"value": d["value"], "unit": "layers/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "qwen2.5-7b-28layer"


def test_bench_help_lists_workloads():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       timeout=120, cwd=ROOT)
    assert r.returncode == 0 and "qwen2.5-14b-48layer-mixed" in r.stdout


def test_traffic_record_keys_ignore_comments(tmp_path, monkeypatch):
    """A DRAM-traffic capture stays valid across comment edits of its kernel source and is
    voided by a code edit."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_text("// header\nint f(int a) {  // trailing\n  /* block\n comment */ return a + 1;\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash("k.cu")
    src.write_text("// header\nint f(int a) {  // trailing\n  /* other\n words */ return a + 1;\n}\n")
    assert bench.source_hash("k.cu") == h0
    src.write_text("// header\nint f(int a) {  // trailing\n  /* block\n comment */ return a + 2;\n}\n")
    assert bench.source_hash("k.cu") != h0


def test_roofline_entry_arithmetic():
    """Workload entries: layers/s, GB/s and the two fractions follow from the elapsed time, the
    step count and the algorithmic bytes per launch."""
    sys.path.insert(0, ROOT)
    import bench
    from qkv_rope_kv_gb300 import configs
    w = configs.QWEN7B
    algo = w.algo_bytes_per_layer()
    e = bench.roofline_entry(w, w.n_layers, 0.5, 1000, w.n_layers, algo)
    assert abs(e["layers_per_s"] - w.n_layers * 1000 / 0.5) < 1e-6
    per_layer = 0.5 / 1000 / w.n_layers
    assert abs(e["hbm_gbs"] - algo / per_layer / 1e9) < 1e-6
    assert abs(e["frac"] - e["hbm_gbs"] / e["peak"]) < 1e-12
    assert abs(e["frac_of_nominal_8000"] - e["hbm_gbs"] / 8000.0) < 1e-12
    assert e["launches_per_step"] == w.n_layers and e["workload"] == w.name


def test_direct_step_only_for_one_plain_layer(monkeypatch):
    """A one-layer decode workload is timed as one qkv_decode_step (or _mixed) launch per step;
    every multi-layer, sweep or fused-norm workload replays its graph (direct_step is None)."""
    import dataclasses
    sys.path.insert(0, ROOT)
    import bench
    import qkv_rope_kv_gb300 as Q
    from qkv_rope_kv_gb300 import configs
    calls = []
    monkeypatch.setattr(Q, "qkv_decode_step", lambda *a: calls.append(("concat", len(a))))
    monkeypatch.setattr(Q, "qkv_decode_step_mixed", lambda *a: calls.append(("mixed", len(a))))
    w = configs.WORKLOADS["qwen2.5-0.5b-single-layer"]
    assert w.n_layers == 1
    layer = dict(x=1, w=2, bias=3, q=4, k=5, v=6, kv_k=7, kv_v=8)
    m = dict(layers=[layer], layer_plans=["plan"], dpos=9)
    bench.direct_step(m, w, "stream")()
    assert calls == [("concat", 11)]
    mixed = dict(x=1, wq=2, wk=3, wv=4, bias_q=5, bias_k=6, bias_v=7, q=8, k=9, v=10, kv_k=11, kv_v=12)
    bench.direct_step(dict(m, layers=[mixed]), w, "stream")()
    assert calls[-1] == ("mixed", 15)
    for other in (configs.QWEN7B, configs.WORKLOADS["qwen2.5-0.5b-24layer-sweep"],
                  dataclasses.replace(w, rmsnorm=True), dataclasses.replace(w, qknorm=True),
                  dataclasses.replace(w, positions=(0, 1))):
        assert bench.direct_step(m, other, "stream") is None
