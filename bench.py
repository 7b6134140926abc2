#!/usr/bin/env python3
"""Throughput of the prefill -> decode KV relayout on GB300.

One step = one whole-prompt hand-off of a batch (every layer, component, head
and token of every prompt: gather through the prefill block table, TP head
re-shard, scatter through the decode block table), one kernel launch through
the C ABI, with the pools resident in HBM. The default workload is the
Llama-3-70B KV shape with one 4096-token prompt, prefill TP4 (block 16) ->
decode TP8 (block 32): 1.34 GB read and 1.34 GB written per step.

Printed: one JSON line (rank 0). ``value`` is the whole-job relayout
throughput in GB/s of algorithmic bytes (read + written), device-timed with
CUDA events over exactly K steps after W warm-up steps, max over ranks.
Extra keys: the per-layer launch mode (eager and CUDA-graph), launches of a
group of layers each (``layer_groups``, CUDA graph), ``e2e`` (the
same metric through the public API with the pools in pinned host memory and
both copies inside the timed region), ``roofline`` (HBM), ``cpu_baseline``
(the CPU oracle on a bounded sample of the same workload) and the SM clocks
sampled during the timed regions.

``--impl reference`` times the CPU oracle instead (the only reference this
method has: the pages ship no implementation of it).

Multi-GPU (torchrun): every rank runs its own replica on its own GPU (the
hand-off of one batch never crosses GPUs); timing is barrier-bracketed and
the slowest rank's time is used, so ``value`` is weak-scaling throughput.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV relayout GB/s (read+write) and % of GB300 HBM peak; ms per 4K-token 70B prompt"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("relayout.cu", "kvr_convert.cuh", "kvr_index.h", "plan.h", "plan.cpp")
WORKLOAD_TEXT = {
    "llama70b": ("Llama-3-70B KV shape: 80 layers, 8 KV heads, head_dim 128, bf16 K/V; "
                 "1 x 4096-token prompt; prefill TP4 (2 heads/shard, block 16) -> decode TP8 "
                 "(1 head/shard, block 32); pools 1.25x the blocks needed"),
    "llama8b": ("Llama-3-8B KV shape: 32 layers, 8 KV heads, head_dim 128, bf16; 16 prompts "
                "U[512,4096]; block 16 -> 32; TP1 -> TP1"),
    "qwen32k": ("Qwen3-32B KV shape: 64 layers, 8 KV heads, head_dim 128, bf16; 4 x 32768 "
                "tokens; prefill TP4 block 16 -> decode TP2 block 64"),
    "qwen32k_ragged": ("Qwen3-32B KV shape, 4 prompts of 32768 - U[1,63] tokens; TP4 block 16 "
                       "-> TP2 block 64"),
    "dsv3mla": ("DeepSeek-V3 MLA latent: 61 layers, one 576-dim bf16 latent per token; 64 "
                "prompts lognormal(median 4096) clipped to [1024, 16384]; block 64 -> 16; TP1"),
    "dsv3mla_tp8": ("DeepSeek-V3 MLA latent replicated over TP8 on both sides: 61 layers, "
                    "576-dim bf16 latent; the first 8 prompts of the dsv3mla draw; block 64 -> "
                    "16; read from the first prefill copy, written to all 8 decode copies"),
    "tiny": "tiny: 2 layers, 2 KV heads, head_dim 64, fp16 bits; 1 x 100 tokens; 16 -> 32",
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="llama70b",
                   choices=["llama70b", "llama8b", "qwen32k", "qwen32k_ragged", "dsv3mla",
                            "dsv3mla_tp8", "tiny"])
    p.add_argument("--layers", type=int, default=None,
                   help="use only the first N layers of the workload (small profiling cases)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=12.0,
                   help="CPU seconds for the oracle baseline sample")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--convert", default="none", choices=["none", "bf16_to_fp8", "fp8_to_bf16"],
                   help="change the KV dtype on the way (FP8 = E4M3, per-head scales)")
    p.add_argument("--sm-sweep", default=None,
                   help="comma-separated SM counts: also time the whole-prompt relayout and "
                        "the ordered per-layer launches on streams limited to that many SMs "
                        "(green contexts); default 16,48,96 for the 70B default run, none "
                        "otherwise; '' for none")
    p.add_argument("--modes", default="all,layer,graph,groups,formats,targets",
                   help="measurements to run: all (whole-prompt, the step), layer (per-layer "
                        "eager launches), graph (per-layer launches replayed from a CUDA "
                        "graph), groups (launches of --groups layers each, from a CUDA graph), "
                        "formats (other decode layouts and the staging-buffer route), "
                        "targets (70B default run: the Qwen3-32B 4 x 32K batch and the 70B "
                        "per-layer conversions, timed like the step), "
                        "overlap (70B, not in the default: the hand-off beside a stand-in for "
                        "the prefill compute; its GEMMs run the GPU at its power limit)")
    p.add_argument("--groups", default="2,4,8,16",
                   help="layers per launch for the groups measurement")
    p.add_argument("--report-windows", action="store_true",
                   help="add the host-clock windows of the timed regions to the line's "
                        "\"run\" entry (targets read them from their child runs)")
    return p.parse_args(argv)


# -- ranks -----------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, local, world


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (x on every rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, steps: int, world: int, max_seconds: float):
    """Aggregate GB/s: every rank moved the same bytes; the slowest rank sets the time."""
    return bytes_per_step_per_rank * steps * world / max_seconds / 1e9


# -- clocks ------------------------------------------------------------------------

CLOCK_FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; kept only for our GPU."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 10:
                continue
            if self.uuid and self.uuid not in parts[1]:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.rows.append(dict(t=ts, sm=float(parts[2]), sm_max=float(parts[3]),
                                      power=_num(parts[4]), active=parts[5],
                                      reasons=dict(zip(REASON_NAMES, parts[6:10]))))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, windows):
        """Median SM clock and the throttle reasons seen inside the given (t0, t1) windows."""
        inside = [r for r in self.rows if any(t0 - 0.05 <= r["t"] <= t1 + 0.05
                                               for t0, t1 in windows)]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi sample fell inside the timed regions"}
        reasons = sorted({k for r in inside for k, v in r["reasons"].items()
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["sm_max"] for r in inside),
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((r["power"] for r in inside if r["power"] is not None),
                                   default=None)}


def _num(s):
    try:
        return float(s)
    except ValueError:
        return None


# -- roofline inputs ----------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "prefill_decode_paged_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config: str, layers: int, suffix: str = ""):
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", f"relayout_{config}{suffix}.md")
    try:
        text = open(path).read()
    except OSError:
        return None, None
    src = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    tr = re.search(r"traffic_bytes_per_full_launch:\s*([0-9]+)", text)
    if not src or not tr or src.group(1) != kernel_source_hash():
        return None, path
    return int(tr.group(1)) * layers // _full_layers(config), path


def _full_layers(config):
    import workloads as wl
    return wl.get(config).num_layers


# -- the CPU oracle -------------------------------------------------------------------

def oracle_sample(w, src_layers, budget_s, reps_cap=1000, conv=None, threads=1):
    """Time the oracle, as it stands, on the given layers of the workload until the
    budget is spent (at least once). Returns (bytes moved, seconds, layers per pass,
    passes). With ``conv`` (the dict given to the plan) the converting oracle runs.
    ``threads`` > 1: each pass splits the layers into that many contiguous ranges and
    runs the oracle on each range in its own host thread (layers write disjoint parts
    of the decode pools; the C call releases the interpreter lock); the pass is timed
    by wall clock."""
    import dataclasses
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    n = len(src_layers[0])
    wk = dataclasses.replace(w, num_layers=n)
    elems = int(w.seq_lens.sum()) * w.num_components * w.kv_heads * w.head_dim
    copies = decode_copies(w)
    if conv is None:
        dst = wk.dst_pools_numpy()
        per_layer = elems * w.elem_bytes * (1 + copies)
    else:
        dst_es = 2 if conv["dst_dtype"] == BF16 else 1
        dst = [np.zeros(wk.dst_shape(), {1: np.uint8, 2: np.uint16}[dst_es])
               for _ in range(wk.dst_tp)]
        per_layer = elems * (w.elem_bytes + dst_es * copies)
        per = w.num_components * (w.kv_heads if conv["per_head"] else 1)   # scales per layer
        geo = wk.geometry()
        geo.pop("elem_bytes")

    def run(lo, hi):
        if conv is None:
            oracle.relayout(src_layers, dst, layer_begin=lo, layer_end=hi, **wk.geometry())
        else:
            oracle.relayout_convert(src_layers, dst, src_dtype=conv["src_dtype"],
                                    dst_dtype=conv["dst_dtype"], per_head=conv["per_head"],
                                    scales=conv["scales"][:per * n], layer_begin=lo,
                                    layer_end=hi, **geo)

    t = max(1, min(threads, n))
    ranges = [(n * k // t, n * (k + 1) // t) for k in range(t)]
    pool = ThreadPoolExecutor(max_workers=t) if t > 1 else None
    moved, spent, reps = 0, 0.0, 0
    try:
        while reps < reps_cap and (reps == 0 or spent < budget_s):
            t0 = time.perf_counter()
            if pool is None:
                run(0, n)
            else:
                for f in [pool.submit(run, lo, hi) for lo, hi in ranges]:
                    f.result()
            spent += time.perf_counter() - t0
            moved += per_layer * n
            reps += 1
    finally:
        if pool is not None:
            pool.shutdown()
    return moved, spent, n, reps


BF16, E4M3 = 1, 2


def conversion(args, w):
    """(prefill workload, decode workload, convert dict or None) for --convert."""
    return conversion_for(args.convert, w)


def conversion_for(kind, w):
    """(prefill workload, decode workload, convert dict or None) for a conversion kind
    ("none", "bf16_to_fp8", "fp8_to_bf16"): FP8 prefill pools hold seeded byte patterns
    spread over every finite E4M3 code (FP8 KV written by a quantizer holds no NaN code),
    scales are seeded per (layer, component, head)."""
    import dataclasses

    import numpy as np
    if kind == "none":
        return w, w, None
    rng = np.random.default_rng(w.seed + 100)
    scales = rng.uniform(0.01, 0.05, w.num_layers * w.num_components * w.kv_heads)
    scales = scales.astype(np.float32)
    fp8 = dataclasses.replace(w, elem_bytes=1, values="e4m3")
    if kind == "bf16_to_fp8":
        return w, fp8, dict(src_dtype=BF16, dst_dtype=E4M3, per_head=True, scales=scales)
    return fp8, w, dict(src_dtype=E4M3, dst_dtype=BF16, per_head=True, scales=scales)


def host_link_ceiling(torch, dev, pairs_in, pairs_out, steps):
    """What the host link gives on the e2e measurement's own pinned buffers: every
    (pinned host, device) pair of ``pairs_in`` copied host -> HBM concurrently with
    every (device, pinned host) pair of ``pairs_out`` copied HBM -> host
    (cudaMemcpyAsync on two streams; wall clock; bytes of both directions)."""
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    moved = sum(h.numel() * h.element_size() for h, _ in pairs_in) + \
        sum(h.numel() * h.element_size() for _, h in pairs_out)

    def once():
        with torch.cuda.stream(up):
            for h, d in pairs_in:
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(down):
            for d, h in pairs_out:
                h.copy_(d, non_blocking=True)
    for _ in range(3):
        once()
    torch.cuda.synchronize(dev)
    rounds = []
    for _ in range(5):      # the copy engines' rate varies between rounds: keep the best
        t0 = time.perf_counter()
        for _ in range(max(1, steps // 2)):
            once()
        torch.cuda.synchronize(dev)
        rounds.append((time.perf_counter() - t0) / max(1, steps // 2))
    sec = min(rounds)
    return {"gbs": round(moved / sec / 1e9, 2), "ms_per_step": round(sec * 1e3, 4),
            "gbs_median": round(moved / statistics.median(rounds) / 1e9, 2),
            "rounds": len(rounds), "bytes_per_step": int(moved),
            "what": "the e2e measurement's pinned pools: every prefill pool host -> HBM "
                    "concurrent with every decode pool HBM -> host (cudaMemcpyAsync, two "
                    "streams)"}


def decode_copies(w):
    """Decode shards that hold each head: Td / H when the decode TP degree exceeds the
    head count (heads replicated), else 1."""
    return max(1, w.dst_tp // w.kv_heads)


def algorithmic_bytes(w, conv):
    """Bytes one whole-prompt hand-off reads plus writes (both arms' metric): every
    head is read once and written to each decode shard that holds it."""
    elems = int(w.seq_lens.sum()) * w.num_layers * w.num_components * w.kv_heads * w.head_dim
    dst_es = w.elem_bytes if conv is None else (2 if conv["dst_dtype"] == BF16 else 1)
    return elems * (w.elem_bytes + dst_es * decode_copies(w))


def dtype_label(w, args, conv):
    if conv is not None:
        return args.convert.replace("_to_", "->")
    return "bf16" if w.values == "randn" else f"u{8 * w.elem_bytes}"


def data_label(w):
    values = "randn bf16 values" if w.values == "randn" else \
        f"random {8 * w.elem_bytes}-bit patterns"
    return f"synthetic (seeded {values} in the prefill pools, seeded random block tables)"


def workload_config(args, w, conv):
    """The ``config`` keys both arms report for the same workload."""
    return {"workload": f"{w.name}: {WORKLOAD_TEXT.get(args.config, args.config)}",
            "mode": "whole-prompt (all layers, one launch per step)",
            "convert": None if conv is None else
            f"{args.convert} (FP8 = E4M3, one scale per layer, component and head)",
            "prompts_per_step": w.num_requests, "tokens_per_step": int(w.seq_lens.sum()),
            "bytes_per_step": algorithmic_bytes(w, conv)}


def host_cpu_model() -> str:
    """The host CPU's model, as the kernel reports it (best effort)."""
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model name"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", text, re.M)
        if m:
            return m.group(1).strip()
    part = re.search(r"^CPU part\s*:\s*(\S+)$", text, re.M)
    impl = re.search(r"^CPU implementer\s*:\s*(\S+)$", text, re.M)
    if part:
        return f"{platform.machine()} (implementer {impl.group(1) if impl else '?'}, " \
               f"part {part.group(1)})"
    return platform.machine()


def host_threads():
    """Host cores this process may run on (the oracle's all-core runs use each once)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


# -- our arm --------------------------------------------------------------------------

def formats_measure(w, src, dev, stream, timed, bytes_step, K, world):
    """The whole-prompt hand-off into other decode layouts, and through a staging
    buffer: head-major decode blocks ([N][H][B][D] per layer and component),
    K and V interleaved per block ([L][N][C][B][H][D] per shard), and the two
    passes of the staging route (pack the prefill pools into [L][C][tokens][H][D],
    pd.py's gathered shape; unpack it into the decode pools), each timed like the
    step. GB/s counts each launch's own bytes read + written."""
    import torch
    from prefill_decode_paged_gb300 import (RelayoutPlan, layout_of_views, pack_plan,
                                            unpack_plan)
    L, C, Nd, Bd, Hd, D = w.dst_shape()
    tdt = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[w.elem_bytes]

    def gbs(ms):
        return round(whole_job_gbs(bytes_step, K, world, ms * 1e-3), 2)

    out = {}
    for name, shape, view in (
            ("head_major", (L, C, Nd, Hd, Bd, D), lambda b, l, c: b[l, c].permute(0, 2, 1, 3)),
            ("kv_interleaved", (L, Nd, C, Bd, Hd, D), lambda b, l, c: b[l, :, c])):
        bufs = [torch.full(shape, -1, dtype=tdt, device=dev) for _ in range(w.dst_tp)]
        views = [[[view(b, l, c) for c in range(C)] for l in range(L)] for b in bufs]
        with RelayoutPlan(src, None, dst_layout=layout_of_views(views), **w.geometry()) as p:
            ms = timed(lambda: p.run_all(stream), K)
        out[name] = {"gbs": gbs(ms), "ms_per_step": round(ms / K, 5)}
        del bufs, views
    total = int(w.seq_lens.sum())
    stage = torch.empty((L, C, total, w.kv_heads, D), dtype=tdt, device=dev)
    dst = w.dst_pools_torch(dev)
    with pack_plan(src, stage, **w.geometry()) as pk, \
            unpack_plan(stage, dst, **w.geometry()) as up:
        ms_p = timed(lambda: pk.run_all(stream), K)
        ms_u = timed(lambda: up.run_all(stream), K)

        def both():
            pk.run_all(stream)
            up.run_all(stream)
        ms_b = timed(both, K)
    out["staging"] = {"pack_gbs": gbs(ms_p), "unpack_gbs": gbs(ms_u),
                      "pack_then_unpack_ms_per_step": round(ms_b / K, 5),
                      "what": "pack: prefill pools -> [L][C][tokens][H][D] staging buffer; "
                              "unpack: staging buffer -> decode pools; each moves the "
                              "prompt's KV once (read + write)"}
    del stage, dst
    torch.cuda.empty_cache()
    return out


def overlap_measure(plan, w, dev, stream, prompts=9):
    """The hand-off beside the prefill compute it belongs to. Stand-in for one layer's
    prefill compute: one bf16 GEMM (cuBLAS) with the FLOPs of a Llama-3-70B layer's
    linear layers for the prompt, [tokens, 8192] x [8192, 104448] (output columns:
    QKV 10240, O 8192, MLP gate and up 57344, down 28672; attention left out).
    Arrangements, per prompt: serial (the L GEMMs, then the whole-prompt hand-off on
    the same stream); layerwise (each layer handed over on a second stream as soon
    as its GEMM is done); layerwise_16sm (the same on a stream limited to 16 SMs).
    Per prompt, events give the span of the GEMMs (first start to last end) and the
    tail: from the last GEMM's end to the end of the hand-off, the time a decode
    instance waits once prefill is done. Medians over `prompts` prompts per
    arrangement, taken in rotation; the GEMM span of each is set beside the GEMMs
    alone with its spread, which bounds how much the hand-off slows the compute."""
    import torch
    from prefill_decode_paged_gb300 import KVRelayoutError, SmStream
    tokens = int(w.seq_lens.sum())
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    a = torch.randn(tokens, 8192, device=dev, dtype=torch.bfloat16, generator=g)
    b = torch.randn(8192, 104448, device=dev, dtype=torch.bfloat16, generator=g) * 0.01
    c = torch.empty(tokens, 104448, device=dev, dtype=torch.bfloat16)
    L = w.num_layers
    side = torch.cuda.Stream(dev)
    done = [torch.cuda.Event() for _ in range(L)]
    try:
        sms = SmStream(16)
    except KVRelayoutError:
        sms = None

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def prompt(kind, handle=None, join=None):
        """One prompt; returns (start, last GEMM end, hand-off end) events."""
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        for layer in range(L):
            torch.mm(a, b, out=c)
            if kind == "layerwise":
                done[layer].record(stream)
                join.wait_event(done[layer])
                plan.run_layer(layer, handle)
        e1.record(stream)
        if kind == "serial":
            plan.run_all(stream)
        elif kind == "layerwise":
            stream.wait_stream(join)
        e2.record(stream)
        return e0, e1, e2

    arrangements = {"compute": lambda: prompt("compute"), "serial": lambda: prompt("serial"),
                    "layerwise": lambda: prompt("layerwise", side, side)}
    if sms is not None:
        ext = torch.cuda.ExternalStream(sms.handle, device=dev)
        arrangements["layerwise_16sm"] = lambda: prompt("layerwise", sms.handle, ext)
    span = {k: [] for k in arrangements}
    tail = {k: [] for k in arrangements}
    with torch.cuda.stream(stream):
        for f in arrangements.values():          # warm-up
            f()
        torch.cuda.synchronize(dev)
        for _ in range(prompts):
            for k, f in arrangements.items():
                e0, e1, e2 = f()
                e2.synchronize()
                span[k].append(e0.elapsed_time(e1))
                tail[k].append(e1.elapsed_time(e2) * 1e3)
    med = statistics.median
    t_c = med(span["compute"])
    out = {"compute_ms": round(t_c, 3),
           "compute_tflops": round(2.0 * tokens * 8192 * 104448 * L / (t_c * 1e-3) / 1e12, 1),
           "compute_spread_ms": round(max(span["compute"]) - min(span["compute"]), 3),
           "tail_us": {k: round(med(v), 1) for k, v in tail.items() if k != "compute"},
           "gemm_span_ms": {k: round(med(v), 3) for k, v in span.items() if k != "compute"},
           "what": "per prompt: stand-in prefill compute (one bf16 GEMM per layer with the "
                   "FLOPs of a 70B layer's linear layers for the prompt); tail = last GEMM's "
                   "end to the hand-off's end; gemm_span = first GEMM's start to last GEMM's "
                   f"end; medians of {prompts} prompts per arrangement"}
    if sms is not None:
        sms.close()
    del a, b, c
    torch.cuda.empty_cache()
    return out


def layer_graph(plan, num_layers, dev, stream, no_wait_after_first=False):
    """The per-layer hand-off of one prompt batch captured once in a CUDA graph:
    ``num_layers`` ordered launches (kv_relayout_layer), or with
    ``no_wait_after_first`` launches 2.. passing KVR_LAUNCH_NO_WAIT (each follows
    another hand-off launch, and every layer is ready before the first)."""
    import torch
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.graph(g, stream=cap):
        for layer in range(num_layers):
            plan.run_layers(layer, 1, wait_for_previous=not no_wait_after_first or layer == 0)
    stream.wait_stream(cap)
    return g


def _figures(bytes_step, ms, steps, world, peak, launches=1):
    """GB/s (whole job), fraction of the copy peak, ms per step and us per launch."""
    gbs = whole_job_gbs(bytes_step, steps, world, ms * 1e-3)
    out = {"gbs": round(gbs, 1), "frac": round(gbs / world / peak, 4),
           "ms": round(ms / steps, 4)}
    if launches > 1:
        out["us_per_launch"] = round(ms * 1e3 / steps / launches, 3)
    return out


def conversion_child(kind, K, W, dev_index):
    """The 70B per-layer conversion ``kind`` timed in a fresh process: ``bench.py
    --convert kind`` (whole prompt and ordered per-layer launches from a CUDA graph,
    K steps each after W warm-up steps) on this rank's GPU alone, its pools the
    first allocations of its CUDA context. Returns (GB/s whole, GB/s per layer, us
    per launch, the child's timed host-clock windows); raises RuntimeError with the
    end of the child's stderr if it fails."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "LOCAL_WORLD_SIZE", "GROUP_RANK",
                        "ROLE_RANK", "MASTER_ADDR", "MASTER_PORT", "TORCHELASTIC_RUN_ID")}
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    env["CUDA_VISIBLE_DEVICES"] = (visible.split(",")[dev_index] if visible
                                   else str(dev_index))
    cmd = [sys.executable, os.path.abspath(__file__), "--config", "llama70b", "--convert", kind,
           "--modes", "all,graph", "--steps", str(K), "--warmup", str(W), "--no-e2e",
           "--no-cpu-baseline", "--no-clocks", "--sm-sweep", "", "--report-windows"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"the {kind} child run failed: {r.stderr.strip()[-400:]}")
    line = json.loads(r.stdout.strip().splitlines()[-1])
    g = line["per_layer"]["cuda_graph"]
    return line["value"], g["gbs"], g["us_per_launch"], line["run"]["timed_windows"]


def targets_measure(timed, dev, stream, K, world, peak, windows, main_per_layer=None):
    """Both >= 80 % targets, and the per-layer hand-off, each timed like the step
    (CUDA events on the launching stream, K steps after warm-up):

    - llama70b per layer with a dtype change on the way (BF16 -> FP8 E4M3 and
      FP8 E4M3 -> BF16, per-head scales): whole prompt, and 80 ordered per-layer
      launches per step (CUDA graph), timed in a fresh process whose pools are its
      first allocations (as an engine allocates its KV cache at start:
      conversion_child); the ordered per-layer launches are timed again in this
      process on pools allocated after the step's own and every earlier
      measurement's (``per_layer_pools_allocated_late``). Where the driver places
      a pool in physical memory moves the ordered BF16 -> FP8 launches by ~5 %;
    - qwen32k: Qwen3-32B KV shape, 4 x 32768 tokens, prefill TP4 block 16 -> decode
      TP2 block 64 (86 GB of pools): one whole-prompt launch per step, and the same
      batch in 64 ordered per-layer launches per step (CUDA graph).

    ``target_ms`` is the time at 80 % of the measured copy peak; ``frac`` is of that
    peak. Each is timed over max(K, 200) steps, at most 2000 (max(K, 30), at most 100,
    for the Qwen batch), after 20 warm-up steps on its freshly allocated pools."""
    import torch

    import workloads as wl
    from prefill_decode_paged_gb300 import RelayoutPlan

    k_big, W = min(max(K, 30), 100), 20
    K = min(max(K, 200), 2000)
    out = {"peak_gbs": peak, "steps": K, "steps_qwen32k": k_big}
    if main_per_layer is not None:
        out["llama70b"] = main_per_layer
    w70 = wl.get("llama70b")
    for kind in ("bf16_to_fp8", "fp8_to_bf16"):
        ws, wd, conv = conversion_for(kind, w70)
        b = algorithmic_bytes(ws, conv)
        # fresh process (each rank its own GPU), then the slowest rank's time; a
        # failed child leaves its figures out (and says why) rather than the line
        try:
            whole_gbs, layer_gbs, _, child_windows = conversion_child(kind, K, W, dev.index)
            windows.extend(tuple(x) for x in child_windows)
            failed = 0.0
        except (RuntimeError, subprocess.TimeoutExpired, ValueError, KeyError) as e:
            whole_gbs = layer_gbs = None
            failed, why = 1.0, str(e)[-400:]
        if max_over_ranks(failed, world, dev) > 0:
            whole = layer = {"error": why if failed else "a child run failed on another rank"}
        else:
            ms_whole = max_over_ranks(b * K / (whole_gbs * 1e9) * 1e3, world, dev)
            ms_layer = max_over_ranks(b * K / (layer_gbs * 1e9) * 1e3, world, dev)
            whole = _figures(b, ms_whole, K, world, peak)
            layer = _figures(b, ms_layer, K, world, peak, ws.num_layers)
        src, dst = ws.src_pools_torch(dev), wd.dst_pools_torch(dev)
        with RelayoutPlan(src, dst, convert=conv, **ws.geometry()) as plan:
            g = layer_graph(plan, ws.num_layers, dev, stream)
            late = _figures(b, timed(g.replay, K, W), K, world, peak, ws.num_layers)
            del g
        out[f"llama70b_{kind}"] = {"whole": whole, "per_layer": layer,
                                   "per_layer_pools_allocated_late": late,
                                   "met": layer.get("frac", 0.0) >= 0.8,
                                   "met_pools_allocated_late": late["frac"] >= 0.8}
        del src, dst
        torch.cuda.empty_cache()
    w = wl.get("qwen32k")
    src, dst = w.src_pools_torch(dev), w.dst_pools_torch(dev)
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        b = plan.bytes_read + plan.bytes_written
        whole = _figures(b, timed(lambda: plan.run_all(stream), k_big, W), k_big, world, peak)
        g = layer_graph(plan, w.num_layers, dev, stream)
        layer = _figures(b, timed(g.replay, k_big, W), k_big, world, peak, w.num_layers)
        del g
    target_ms = b / (0.8 * peak * 1e9) * 1e3
    out["qwen32k"] = {"whole": whole, "per_layer": layer, "target_ms": round(target_ms, 3),
                      "met": whole["ms"] <= target_ms and layer["ms"] <= target_ms}
    del src, dst
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import numpy as np
    import torch

    import workloads as wl
    from prefill_decode_paged_gb300 import RelayoutPlan

    rank, local, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the relayout only runs on the GPU")
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)

    w = wl.get(args.config)
    if args.layers:
        w = w.with_layers(args.layers)
    w, w_dst, conv = conversion(args, w)
    src = w.src_pools_torch(dev)
    dst = w_dst.dst_pools_torch(dev)
    plan = RelayoutPlan(src, dst, convert=conv, **w.geometry())
    bytes_step = plan.bytes_read + plan.bytes_written
    if bytes_step != algorithmic_bytes(w, conv):
        raise SystemExit("bench.py: the plan's byte count differs from the workload's")
    stream = torch.cuda.current_stream(dev)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    windows = []

    def timed(fn, steps, warmup=None):
        for _ in range(args.warmup if warmup is None else warmup):
            fn()
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        t_host = time.time()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        windows.append((t_host, time.time()))
        ms = ev0.elapsed_time(ev1)
        barrier(world)
        return max_over_ranks(ms, world, dev)

    K = args.steps
    # whole-prompt: one launch per step
    ms_all = timed(lambda: plan.run_all(stream), K)
    # single launches: 20 whole-prompt launches, each timed alone (median, best)
    singles = []
    for _ in range(20):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        plan.run_all(stream)
        e1.record(stream)
        e1.synchronize()
        singles.append(e0.elapsed_time(e1))
    launch_ms = {"median": round(statistics.median(singles), 5), "best": round(min(singles), 5),
                 "samples": len(singles)}
    modes = set(args.modes.split(","))
    L = w.num_layers
    ms_layer = ms_graph = ms_graph_nw = None
    k_layer = max(1, K // 4)
    if "layer" in modes:
        # per-layer, eager: L launches per step from Python
        def per_layer():
            for layer in range(L):
                plan.run_layer(layer, stream)
        ms_layer = timed(per_layer, k_layer)
    if "graph" in modes:
        # per-layer, the L launches captured once in a CUDA graph and replayed
        g = layer_graph(plan, L, dev, stream)
        ms_graph = timed(g.replay, K)
        del g
        # the same launches where each but the first passes KVR_LAUNCH_NO_WAIT: they
        # follow another hand-off launch and their layers are ready before it (all are)
        g = layer_graph(plan, L, dev, stream, no_wait_after_first=True)
        ms_graph_nw = timed(g.replay, K)
        del g
    layer_groups = None
    if "groups" in modes:
        # layer groups: ceil(L / n) launches of n layers each (kv_relayout_layers), the
        # way an engine that computes prefill n layers per round would hand KV over;
        # captured in a CUDA graph like the per-layer launches
        layer_groups = {}
        for n in [int(x) for x in args.groups.split(",") if x]:
            if n < 2 or n >= L:
                continue
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.graph(g, stream=cap):
                for first in range(0, L, n):
                    plan.run_layers(first, min(n, L - first))
            stream.wait_stream(cap)
            ms = timed(g.replay, K)
            launches = -(-L // n)
            layer_groups[str(n)] = {
                "gbs": round(whole_job_gbs(bytes_step, K, world, ms * 1e-3), 2),
                "ms_per_prompt": round(ms / K / w.num_requests, 5),
                "us_per_launch": round(ms * 1e3 / K / launches, 3),
                "launches_per_step": launches}
            del g

    # other decode layouts and the staging-buffer route (70B workload, bit copy)
    formats = None
    if "formats" in modes and args.config == "llama70b" and conv is None and not args.layers:
        formats = formats_measure(w, src, dev, stream, timed, bytes_step, K, world)

    # the whole-prompt relayout on streams limited to a number of SMs
    sm_sweep = None
    sweep_spec = args.sm_sweep
    if sweep_spec is None:
        sweep_spec = "16,48,96" if (args.config == "llama70b" and conv is None and
                                    not args.layers) else ""
    if sweep_spec:
        from prefill_decode_paged_gb300 import KVRelayoutError, SmStream
        sm_sweep = {}
        for want in [int(x) for x in sweep_spec.split(",") if x]:
            try:
                sms = SmStream(want)
            except KVRelayoutError as e:      # no green contexts here: say so, go on
                sm_sweep[str(want)] = {"unavailable": e.name}
                continue
            with sms:
                ext = torch.cuda.ExternalStream(sms.handle, device=dev)
                steps = max(1, K // 4)
                for _ in range(3):
                    plan.run_all(sms.handle)
                ext.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                th = time.time()
                e0.record(ext)
                for _ in range(steps):
                    plan.run_all(sms.handle)
                e1.record(ext)
                ext.synchronize()
                windows.append((th, time.time()))
                ms = e0.elapsed_time(e1) / steps
                # the same hand-off layer by layer (L ordered launches per step)
                for layer in range(L):
                    plan.run_layer(layer, sms.handle)
                ext.synchronize()
                th = time.time()
                e0.record(ext)
                for _ in range(steps):
                    for layer in range(L):
                        plan.run_layer(layer, sms.handle)
                e1.record(ext)
                ext.synchronize()
                windows.append((th, time.time()))
                ms_l = e0.elapsed_time(e1) / steps
                sm_sweep[str(sms.sms)] = {"gbs": round(bytes_step / (ms * 1e-3) / 1e9, 1),
                                          "ms_per_step": round(ms, 4),
                                          "per_layer_gbs": round(
                                              bytes_step / (ms_l * 1e-3) / 1e9, 1)}

    hbm_peak, peak_src = measured_hbm_peak()

    # both >= 80 % targets and the per-layer conversions (the default 70B run only)
    targets = None
    if "targets" in modes and args.config == "llama70b" and conv is None and not args.layers:
        main = None
        if ms_graph is not None:
            main = {"whole": _figures(bytes_step, ms_all, K, world, hbm_peak),
                    "per_layer": _figures(bytes_step, ms_graph, K, world, hbm_peak, L),
                    "target_ms": round(bytes_step / (0.8 * hbm_peak * 1e9) * 1e3, 4)}
            main["met"] = max(main["whole"]["ms"], main["per_layer"]["ms"]) <= main["target_ms"]
        targets = targets_measure(timed, dev, stream, K, world, hbm_peak, windows, main)

    # e2e: the pools live in pinned host memory; every step hands the batch over
    # through the public no-allocation call, whose kernel reads the prefill rows
    # from host memory and writes the decode rows to host memory over
    # NVLink-C2C (inputs host -> device and results device -> host inside the
    # kernel), then waits for it. The staged variant (copy the whole pools to
    # HBM, plan, relayout, copy the decode pools back) is reported beside it.
    e2e = e2e_staged = None
    pinned_budget = 16 << 30
    pool_bytes = sum(t.numel() * t.element_size() for t in src + dst)
    if not args.no_e2e and pool_bytes <= pinned_budget and conv is None:
        from prefill_decode_paged_gb300 import relayout_all_prealloc
        h_src = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in src]
        h_dst = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dst]
        for h, t in zip(h_src, src):
            h.copy_(t)
        for h in h_dst:
            h.fill_(-1)
        # the work list the call copies to the device: 16 B per token tile (here one
        # decode block), 8 B per (shard, layer, component) view base of each side, 4 B
        # per used prefill and decode block id
        meta_bytes = 16 * sum(-(-int(n) // w.dst_block) for n in w.seq_lens) + \
            8 * (w.src_tp + w.dst_tp) * w.num_layers * w.num_components + \
            4 * sum(-(-int(n) // w.src_block) + -(-int(n) // w.dst_block) for n in w.seq_lens)

        def run_e2e(step, steps, what, h2d, d2h):
            for _ in range(min(args.warmup, 3)):
                step()
            torch.cuda.synchronize(dev)
            barrier(world)
            t0 = time.perf_counter()
            th = time.time()
            for _ in range(steps):
                step()
            torch.cuda.synchronize(dev)
            sec = time.perf_counter() - t0
            windows.append((th, time.time()))
            barrier(world)
            sec = max_over_ranks(sec, world, dev)
            return {"value": round(whole_job_gbs(bytes_step, steps, world, sec), 2),
                    "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "steps": steps,
                    "ms_per_step": round(sec * 1e3 / steps, 4), "what": what}

        def zero_copy_step():
            relayout_all_prealloc(h_src, h_dst, stream, **w.geometry())
            torch.cuda.synchronize(dev)

        e2e = run_e2e(zero_copy_step, args.e2e_steps,
                      "per step: kv_relayout_all_prealloc on pools in pinned host memory "
                      "(the kernel reads and writes them over NVLink-C2C), synchronize; "
                      "wall clock",
                      plan.bytes_read + meta_bytes, plan.bytes_written)
        for h, t in zip(h_dst, dst):
            if not torch.equal(h.to(dev), t):
                raise SystemExit("bench.py: host-pool relayout differs from the HBM one")
        e2e["link_ceiling"] = host_link_ceiling(torch, dev, list(zip(h_src, src)),
                                                list(zip(dst, h_dst)), args.e2e_steps)
        e2e["frac_of_link"] = round(e2e["value"] / e2e["link_ceiling"]["gbs"], 4)

        def staged_step():
            for h, t in zip(h_src, src):
                t.copy_(h, non_blocking=True)
            with RelayoutPlan(src, dst, **w.geometry()) as p:
                p.run_all(stream)
                for h, t in zip(h_dst, dst):
                    h.copy_(t, non_blocking=True)
                torch.cuda.synchronize(dev)

        e2e_staged = run_e2e(
            staged_step, args.e2e_steps,
            "per step: pinned-host -> HBM copy of every prefill shard pool, "
            "kv_relayout_plan, kv_relayout_all, HBM -> pinned-host copy of every decode "
            "shard pool, synchronize; wall clock",
            sum(t.numel() * t.element_size() for t in h_src) + meta_bytes,
            sum(t.numel() * t.element_size() for t in h_dst))
        del h_src, h_dst

    clock = None
    if clocks:
        time.sleep(0.25)
        clocks.stop()
        clock = clocks.summary(windows)

    # the per-layer hand-off beside the prefill compute it belongs to (70B workload);
    # after the clock record: its GEMMs run the GPU at its power limit, which would
    # otherwise show in the throttle reasons of the timed regions next to it
    overlap = None
    if "overlap" in modes and args.config == "llama70b" and conv is None and not args.layers:
        overlap = overlap_measure(plan, w, dev, stream)

    # CPU oracle on a bounded sample (rank 0, N = 1 only): on every host core (one
    # thread per core, each on its own range of layers), and on one core
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = host_threads()
        n_layers = max(1, min(L, max(8, cores)))
        src_layers = [np.ascontiguousarray(t[:n_layers].cpu().numpy().view(w.int_dtype()))
                      for t in src]
        moved, sec, nl, reps = oracle_sample(w, src_layers, args.cpu_budget_s * 2 / 3,
                                             conv=conv, threads=cores)
        used = min(cores, nl)
        one = [a[:min(nl, 8)] for a in src_layers]
        moved1, sec1, nl1, reps1 = oracle_sample(w, one, args.cpu_budget_s / 3, conv=conv)
        cpu = {"value": round(moved / sec / 1e9, 4), "unit": "GB/s", "cores": used,
               "kind": "oracle",
               "sample": f"{reps} pass(es) of the oracle over the first {nl} of {L} layers of "
                         f"the same workload, {used} host threads each on its own range of "
                         f"layers ({moved} bytes read+written in {sec:.1f} s), host copies of "
                         f"the same prefill pools",
               "single_thread": {"value": round(moved1 / sec1 / 1e9, 4), "cores": 1,
                                 "sample": f"{reps1} pass(es) over the first {nl1} layers "
                                           f"({moved1} bytes in {sec1:.1f} s)"},
               "host_cpus": os.cpu_count(), "host_cpu": host_cpu_model()}

    avg_launch_ms = ms_all / K
    achieved = bytes_step / (avg_launch_ms * 1e-3) / 1e9
    traffic, _ = profiled_traffic(args.config, w.num_layers,
                                  "" if conv is None else f"_{args.convert}")
    prompts = w.num_requests
    value = whole_job_gbs(bytes_step, K, world, ms_all * 1e-3)

    def per_layer_entry(ms, steps, extra=None):
        if ms is None:
            return None
        e = {"gbs": round(whole_job_gbs(bytes_step, steps, world, ms * 1e-3), 2),
             "ms_per_prompt": round(ms / steps / prompts, 5),
             "us_per_launch": round(ms * 1e3 / steps / L, 3)}
        return {**e, **(extra or {})}

    # key order: the driver keeps the end of stdout, so the per-layer figures and the
    # targets come last
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_all / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_label(w, args, conv),
        "data": data_label(w),
        "config": workload_config(args, w, conv),
        "run": {"l2": "inputs larger than L2 (no flush)" if bytes_step > 2 * 129e6 else
                      "working set fits in L2 (launch-bound case)",
                "parallelism": f"replica per GPU x{world}", "impl": "CUDA kernel via the C ABI",
                **({"timed_windows": [[round(a, 3), round(b, 3)] for a, b in windows]}
                   if args.report_windows else {})},
        "ms_per_prompt": round(ms_all / K / prompts, 5),
        "launch_ms": launch_ms,
        "pct_of_hbm_peak": round(100 * achieved / hbm_peak, 2),
        "pct_of_nominal_hbm": round(100 * achieved / NOMINAL_HBM_GBS, 2),
        "gpu_launches": K,
        "formats": formats,
        "overlap": overlap,
        "layer_groups": layer_groups,
        "sm_sweep": sm_sweep,
        "e2e_staged": e2e_staged,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": traffic, "peak_source": f"{peak_src} (copy, read+write)",
                     "kernel": "kvr_relayout_kernel",
                     "algorithmic_bytes_per_launch": bytes_step},
        "clocks": clock,
        "per_layer": {
            "launches_per_step": L,
            "eager": per_layer_entry(ms_layer, k_layer),
            "cuda_graph": per_layer_entry(ms_graph, K),
            "cuda_graph_no_wait": per_layer_entry(ms_graph_nw, K,
                                                  {"what": "launches 2..L pass "
                                                           "KVR_LAUNCH_NO_WAIT"}),
        },
        "targets": targets,
    }
    plan.close()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# -- reference arm: the CPU oracle ----------------------------------------------------------

def run_reference(args):
    import numpy as np

    import workloads as wl
    rank, local, world = dist_env()
    if rank != 0:
        return
    w = wl.get(args.config)
    if args.layers:
        w = w.with_layers(args.layers)
    w, _, conv = conversion(args, w)
    # per step: a bounded sample of layers, sized so W + K steps take about two minutes,
    # run on every host core (one thread per core, each on its own range of layers)
    cores = host_threads()
    probe = w.with_layers(1)
    src1 = probe.src_pools_numpy()
    _, t1, _, _ = oracle_sample(probe, [a for a in src1], 0.0, reps_cap=1, conv=conv)
    per_layer_s = max(t1, 1e-4)
    total = args.steps + args.warmup
    n = int(max(1, min(w.num_layers, 120.0 * cores / (total * per_layer_s))))
    wk = w.with_layers(n)
    src = wk.src_pools_numpy()
    for _ in range(args.warmup):
        oracle_sample(wk, src, 0.0, reps_cap=1, conv=conv, threads=cores)
    moved, spent = 0, 0.0
    for _ in range(args.steps):
        m, s, _, _ = oracle_sample(wk, src, 0.0, reps_cap=1, conv=conv, threads=cores)
        moved += m
        spent += s
    gbs = moved / spent / 1e9
    step_ms = spent * 1e3 / args.steps
    used = min(cores, n)
    cpu = {"value": round(gbs, 4), "unit": "GB/s", "kind": "oracle", "cores": used,
           "sample": f"each step: the oracle over the first {n} of {w.num_layers} layers of the "
                     f"workload (all prompts, all heads), {used} host threads each on its own "
                     f"range of layers", "host_cpus": os.cpu_count(),
           "host_cpu": host_cpu_model()}
    out = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(step_ms, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": dtype_label(w, args, conv),
           "data": data_label(w),
           "config": workload_config(args, w, conv),
           "run": {"sample_layers_per_step": n,
                   "parallelism": f"CPU oracle, {used} host threads", "impl": "CPU oracle"},
           "cpu_baseline": cpu,
           "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
