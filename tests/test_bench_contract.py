"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
fp64 oracle on a bounded sample of the workload and prints one JSON line with
the same metric, unit and config as the GPU arm; under torchrun only rank 0
prints it, and the other ranks exit 0 without work."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ, **(extra_env or {}))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--ref-step-s", "0.5"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_line():
    lines = _run()
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("mid_causal:")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == "TFLOP/s" and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # ms_per_step is the workload's FLOPs at the measured rate
    fl = sum(bench.workload_flops(*_workload_args()))
    assert abs(d["ms_per_step"] - fl / (d["value"] * 1e12) * 1e3) <= 1e-6 * d["ms_per_step"]


def _workload_args():
    import synth
    w = synth.workloads()["mid_causal"]
    inp = synth.make_workload(w)
    return w, inp["lengths"], inp.get("lengths_k")


def test_reference_arm_other_rank_is_silent():
    assert _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_traffic_figure_is_tied_to_the_kernel_sources(monkeypatch):
    """roofline.traffic is the recorded DRAM bytes only while the backward's
    sources are the ones the capture was taken on; otherwise null."""
    import bench
    sha = bench.sources_sha()
    monkeypatch.setattr(bench, "FA_BWD_DRAM", {"mid_causal": {"bytes": 1.0e9, "sources": sha}})
    assert bench.bwd_traffic("mid_causal") == 1.0e9
    assert bench.bwd_traffic("long_causal") is None
    monkeypatch.setattr(bench, "FA_BWD_DRAM",
                        {"mid_causal": {"bytes": 1.0e9, "sources": "0" * 16}})
    assert bench.bwd_traffic("mid_causal") is None


def test_steps_for_fills_the_clock_window():
    import bench
    # a 0.34 ms step plus the flush: about 2 s of steps
    assert 4000 <= bench.steps_for(0.34, 2.0, lo=200) <= 5000
    assert bench.steps_for(100.0, 1.0, lo=10) == 10


def test_traffic_hash_ignores_comments_not_code(tmp_path):
    """A comment or layout edit keeps the recorded traffic; a code edit drops it."""
    import bench
    src = 'int f(int a) {  // one\n  /* two */ return a + 1; }\nconst char* s = "x//y";\n'
    variants = {
        "base": src,
        "comment": src.replace("// one", "// another comment").replace("/* two */", ""),
        "layout": src.replace("  return", "\n\n        return"),
        "code": src.replace("a + 1", "a + 2"),
        "string": src.replace("x//y", "x//z"),
    }
    sha = {}
    for k, text in variants.items():
        f = tmp_path / f"{k}.cu"
        f.write_text(text)
        sha[k] = bench.sources_sha([str(f)])
    assert sha["comment"] == sha["base"] and sha["layout"] == sha["base"]
    assert sha["code"] != sha["base"] and sha["string"] != sha["base"]
