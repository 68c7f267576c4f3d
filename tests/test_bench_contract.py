"""The benchmark's reference arm (the CPU oracle timed on the host cores) runs
on the CPU and prints one JSON line with every key the benchmark contract
asks for; its metric, unit and direction are the GPU arm's."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["unit"] == "GB/s" and d["dtype"] == "f64" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert d["vs_baseline"] is None


def test_traffic_figure_belongs_to_the_current_kernel_sources():
    """The bench line's roofline.traffic is a DRAM byte count taken with ncu
    from the kernels as they are; it is keyed to a hash of the kernel sources.
    A kernel edit without a new capture would silently null the figure, so a
    stale key fails here: re-run the DRAM metrics pass over the step's four
    launch kinds and update bench.TRAFFIC."""
    import importlib.util

    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.TRAFFIC["csrc_sha"] == bench.csrc_sha(), (bench.TRAFFIC["csrc_sha"], bench.csrc_sha())
    assert bench.TRAFFIC["bytes_per_launch"] > 0
