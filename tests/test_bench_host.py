"""bench.py host logic on the CPU: rank aggregation over gloo, the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    slowest = bench.max_over_ranks(1.0 + rank, world)       # rank r took 1 + r seconds
    gbs = bench.whole_job_gbs(10**9, 4, world, slowest)
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump({"max": slowest, "gbs": gbs}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    out = str(tmp_path / "r")
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        with open(f"{out}.{r}") as f:
            got = json.load(f)
        assert got["max"] == 2.0
        # 2 ranks x 4 steps x 1 GB over the slowest rank's 2 s
        assert got["gbs"] == pytest.approx(4.0)


def test_reference_arm_prints_the_contract_line():
    sys.path.insert(0, ROOT)
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "3", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "cpu_baseline", "e2e", "config"):
        assert k in d, k
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    # the workload's config only; how the arm ran goes under "run"
    import bench
    import workloads as wl
    args = bench.parse_args(["--impl", "reference", "--config", "tiny"])
    assert d["config"] == bench.workload_config(args, wl.get("tiny"), None)
    assert "sample_layers_per_step" in d["run"]


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_traffic_is_dropped_when_the_kernel_changed(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "relayout_llama70b.md").write_text(
        "kernel_source_sha256: 0000000000000000\ntraffic_bytes_per_full_launch: 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "prefill_decode_paged_gb300" / "csrc")
    for name in bench.KERNEL_SOURCES:
        src = os.path.join(ROOT, "prefill_decode_paged_gb300", "csrc", name)
        with open(src, "rb") as f, open(tmp_path / "prefill_decode_paged_gb300" / "csrc" / name,
                                        "wb") as g:
            g.write(f.read())
    assert bench.profiled_traffic("llama70b", 80)[0] is None
    h = bench.kernel_source_hash()
    (prof / "relayout_llama70b.md").write_text(
        f"kernel_source_sha256: {h}\ntraffic_bytes_per_full_launch: 8000\n")
    assert bench.profiled_traffic("llama70b", 80)[0] == 8000
    assert bench.profiled_traffic("llama70b", 8)[0] == 800


@pytest.mark.parametrize("name", ["llama70b", "qwen32k", "dsv3mla", "dsv3mla_tp8"])
@pytest.mark.parametrize("convert", [None, "bf16_to_fp8"])
def test_bench_bytes_equal_the_librarys_count(name, convert):
    """bench.py cross-checks the plan's byte count against its own workload arithmetic;
    the two must agree for every named workload (replicated decode copies included)."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    from prefill_decode_paged_gb300 import kv_relayout as kr
    w = wl.get(name)
    base, gap, s, d = 1 << 40, 1 << 20, [], []
    at = base
    for _ in range(w.src_tp):
        s.append(at)
        at += (w.src_pool_bytes() + gap) // 256 * 256 + 256
    dst_es = 1 if convert else w.elem_bytes
    for _ in range(w.dst_tp):
        d.append(at)
        at += (w.dst_pool_bytes() * dst_es // w.elem_bytes + gap) // 256 * 256 + 256
    conv = None
    if convert:
        import numpy as np
        conv = dict(src_dtype=bench.BF16, dst_dtype=2, per_head=0,
                    scales=np.ones(w.num_layers * w.num_components, np.float32))
    r, wr = kr.desc_bytes(s, d, convert=conv, **w.geometry())
    assert r + wr == bench.algorithmic_bytes(w, conv)


def test_conversion_targets_run_in_a_fresh_single_gpu_process(monkeypatch):
    """The targets' conversion runs are bench.py children on this rank's GPU alone:
    no rank variables, the rank's device as the only visible one, and their whole,
    per-layer and timed-window figures read back from the child's line."""
    sys.path.insert(0, ROOT)
    import bench
    seen = {}

    def fake_run(cmd, env, capture_output, text, timeout):
        seen.update(cmd=cmd, env=env)
        line = {"value": 7000.0, "per_layer": {"cuda_graph": {"gbs": 5600.0,
                                                              "us_per_launch": 4.5}},
                "run": {"timed_windows": [[1.0, 2.0], [3.0, 4.0]]}}
        return subprocess.CompletedProcess(cmd, 0, stdout="noise\n" + json.dumps(line) + "\n",
                                           stderr="")

    monkeypatch.setattr(bench.subprocess, "run", fake_run)
    for k, v in dict(RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                     MASTER_PORT="29500", CUDA_VISIBLE_DEVICES="4,5").items():
        monkeypatch.setenv(k, v)
    whole, layer, us, windows = bench.conversion_child("bf16_to_fp8", 200, 20, 1)
    assert (whole, layer, us, windows) == (7000.0, 5600.0, 4.5, [[1.0, 2.0], [3.0, 4.0]])
    env, cmd = seen["env"], seen["cmd"]
    assert not {"RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT"} & set(env)
    assert env["CUDA_VISIBLE_DEVICES"] == "5"
    assert cmd[cmd.index("--convert") + 1] == "bf16_to_fp8"
    assert cmd[cmd.index("--steps") + 1] == "200" and cmd[cmd.index("--warmup") + 1] == "20"
    assert "--report-windows" in cmd and cmd[cmd.index("--modes") + 1] == "all,graph"
    # a failed child raises with the end of its stderr (targets_measure records it)
    monkeypatch.setattr(bench.subprocess, "run", lambda cmd, **kw: subprocess.CompletedProcess(
        cmd, 1, stdout="", stderr="boom"))
    with pytest.raises(RuntimeError, match="boom"):
        bench.conversion_child("fp8_to_bf16", 200, 20, 0)
