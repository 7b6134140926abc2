"""bench.py on the GPU: the JSON line keeps its contract (small workload, few steps)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keeps_the_contract():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--config", "tiny",
                          "--steps", "20", "--warmup", "3", "--e2e-steps", "3",
                          "--cpu-budget-s", "0.2"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "gpu_launches", "roofline", "e2e", "cpu_baseline", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3
    assert d["gpu_launches"] == 20
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["bytes_per_step"] == 204800
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    # tiny has 2 layers: at most 2 threads, each on its own layer; and the one-core figure
    assert c["cores"] <= 2 and c["single_thread"]["cores"] == 1
    assert c["single_thread"]["value"] > 0
    assert d["per_layer"]["launches_per_step"] == 2
    assert d["per_layer"]["eager"]["gbs"] > 0 and d["per_layer"]["cuda_graph"]["gbs"] > 0
    # the reference arm reports the identical config for the same workload
    ref = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "3", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert ref.returncode == 0, ref.stderr[-3000:]
    assert json.loads(ref.stdout.strip().splitlines()[-1])["config"] == d["config"]
    # the per-layer figures and the targets close the line (the end of stdout is what
    # a log tail keeps)
    assert list(d)[-2:] == ["per_layer", "targets"]
