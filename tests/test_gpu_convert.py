"""GPU parity of the converting relayout (BF16 <-> FP8 E4M3) against the CPU oracle.

Bit-exact: both sides compute the same fp32 product and round it the same
way, so every code and every BF16 pattern must match, including NaN, signed
zeros, saturated values and subnormals (the inputs are uniform random bit
patterns besides N(0,1) data).
"""
import dataclasses
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from prefill_decode_paged_gb300 import RelayoutPlan
from prefill_decode_paged_gb300.kv_relayout import DTYPE_BF16, DTYPE_FP8_E4M3

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    import gc
    import torch
    gc.collect()
    torch.cuda.empty_cache()


def _geometry(w):
    g = w.geometry()
    g.pop("elem_bytes")
    return g


def _scales(rng, w, per_head, lo=0.004, hi=2.0):
    n = w.num_layers * w.num_components * (w.kv_heads if per_head else 1)
    return rng.uniform(lo, hi, n).astype(np.float32)


def _src_bits(rng, w, dtype, randn_scale=None):
    out = []
    for _ in range(w.src_tp):
        if dtype == DTYPE_BF16:
            if randn_scale is None:
                out.append(rng.integers(0, 1 << 16, w.src_shape(), dtype=np.uint16))
            else:
                f = (rng.standard_normal(w.src_shape(), dtype=np.float32) * randn_scale)
                u = f.view(np.uint32)
                out.append(((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16))
        else:
            out.append(rng.integers(0, 256, w.src_shape(), dtype=np.uint8))
    return out


def _dst(w, dtype):
    dt = np.uint16 if dtype == DTYPE_BF16 else np.uint8
    fill = 0xFFFF if dtype == DTYPE_BF16 else 0xFF
    return [np.full(w.dst_shape(), fill, dt) for _ in range(w.dst_tp)]


def _to_dev(arrays):
    import torch
    return [torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
            for a in arrays]


def _run_gpu(w, src_np, dst_np, conv, mode):
    import torch
    src, dst = _to_dev(src_np), _to_dev(dst_np)
    with RelayoutPlan(src, dst, convert=conv, **w.geometry()) as plan:
        if mode == "all":
            plan.run_all()
        elif mode == "layer":
            for layer in range(w.num_layers):
                plan.run_layer(layer)
        else:                                  # layer ranges
            plan.run_layers(0, w.num_layers - 1)
            plan.run_layers(w.num_layers - 1, 1)
        torch.cuda.synchronize()
    return [t.cpu().numpy().view(a.dtype) for t, a in zip(dst, dst_np)]


def _check(w, src_np, src_dtype, dst_dtype, per_head, scales, modes=("all", "layer")):
    ref = _dst(w, dst_dtype)
    oracle.relayout_convert(src_np, ref, src_dtype=src_dtype, dst_dtype=dst_dtype,
                            per_head=per_head, scales=scales, **_geometry(w))
    conv = dict(src_dtype=src_dtype, dst_dtype=dst_dtype, per_head=per_head, scales=scales)
    for mode in modes:
        got = _run_gpu(w, src_np, _dst(w, dst_dtype), conv, mode)
        for s, (a, b) in enumerate(zip(ref, got)):
            if not np.array_equal(a, b):
                bad = np.argwhere(a != b)[:5]
                raise AssertionError(f"{w.name} {mode} shard {s}: {len(np.argwhere(a != b))} "
                                     f"mismatches, first at {bad.tolist()}: "
                                     f"want {a[tuple(bad[0])]:#x} got {b[tuple(bad[0])]:#x}")


SMALL = {
    "tp4_to_tp8": dict(num_layers=3, num_components=2, kv_heads=8, head_dim=16, src_tp=4,
                       dst_tp=8, src_block=16, dst_block=32, seq_lens=[300, 1, 33]),
    "tp4_to_tp2_16_64": dict(num_layers=2, num_components=2, kv_heads=8, head_dim=32, src_tp=4,
                             dst_tp=2, src_block=16, dst_block=64, seq_lens=[695, 637, 64, 65]),
    "mla_64_16": dict(num_layers=2, num_components=1, kv_heads=1, head_dim=576, src_tp=1,
                      dst_tp=1, src_block=64, dst_block=16, seq_lens=[129, 64, 1000]),
    "tp3_to_tp2_odd": dict(num_layers=2, num_components=2, kv_heads=6, head_dim=48, src_tp=3,
                           dst_tp=2, src_block=3, dst_block=5, seq_lens=[40, 0, 17, 1]),
    "block_1_to_64": dict(num_layers=1, num_components=2, kv_heads=4, head_dim=128, src_tp=1,
                          dst_tp=4, src_block=1, dst_block=64, seq_lens=[1000, 63]),
    # replicated heads: a per-head scale belongs to the head, whichever copy holds it
    "rep_h2_tp8_to_tp16": dict(num_layers=2, num_components=2, kv_heads=2, head_dim=32,
                               src_tp=8, dst_tp=16, src_block=16, dst_block=5,
                               seq_lens=[77, 16]),
    "mla_tp2_to_tp4": dict(num_layers=2, num_components=1, kv_heads=1, head_dim=576, src_tp=2,
                           dst_tp=4, src_block=64, dst_block=16, seq_lens=[129, 1]),
}


@pytest.mark.parametrize("per_head", [0, 1])
@pytest.mark.parametrize("case", sorted(SMALL))
def test_quantize_random_bits(case, per_head):
    rng = np.random.default_rng(zlib.crc32(case.encode()) % 1000 + per_head)
    w = wl.custom(case, 300 + per_head, elem_bytes=2, **SMALL[case])
    _check(w, _src_bits(rng, w, DTYPE_BF16), DTYPE_BF16, DTYPE_FP8_E4M3, per_head,
           _scales(rng, w, per_head))


@pytest.mark.parametrize("per_head", [0, 1])
@pytest.mark.parametrize("case", sorted(SMALL))
def test_dequantize_random_codes(case, per_head):
    rng = np.random.default_rng(zlib.crc32(case.encode()) % 1000 + 7 + per_head)
    w = wl.custom(case, 400 + per_head, elem_bytes=1, **SMALL[case])
    _check(w, _src_bits(rng, w, DTYPE_FP8_E4M3), DTYPE_FP8_E4M3, DTYPE_BF16, per_head,
           _scales(rng, w, per_head, 0.5, 1e3))


def test_quantize_typical_values_and_tiny_huge_scales():
    rng = np.random.default_rng(11)
    w = wl.custom("typ", 12, elem_bytes=2, **SMALL["tp4_to_tp8"])
    src = _src_bits(rng, w, DTYPE_BF16, randn_scale=0.3)
    for scales in (_scales(rng, w, 0, 0.001, 0.01),       # many saturated codes
                   _scales(rng, w, 0, 10.0, 500.0),       # many subnormal codes and zeros
                   np.full(w.num_layers * 2, 1.0 / 448, np.float32)):
        _check(w, src, DTYPE_BF16, DTYPE_FP8_E4M3, 0, scales, modes=("all",))


def test_llama70b_quantize_full_size_every_layer():
    """The 70B workload relaid into an FP8 decode pool: the whole-prompt launch against
    the oracle on every layer (one host thread per layer at a time: the converting
    oracle takes about a second per layer), and the per-layer launches equal to it."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import torch
    w = wl.llama70b()
    rng = np.random.default_rng(70)
    scales = _scales(rng, w, 1, 0.002, 0.02)
    conv = dict(src_dtype=DTYPE_BF16, dst_dtype=DTYPE_FP8_E4M3, per_head=1, scales=scales)
    src = w.src_pools_torch("cuda")
    dst = [torch.full(w.dst_shape(), 0xFF, dtype=torch.uint8, device="cuda")
           for _ in range(w.dst_tp)]
    with RelayoutPlan(src, dst, convert=conv, **w.geometry()) as plan:
        assert plan.bytes_read == 1_342_177_280 and plan.bytes_written == 671_088_640
        plan.run_all()
        torch.cuda.synchronize()
    w1 = dataclasses.replace(w, num_layers=1)
    src_host = [t.cpu().numpy().view(np.uint16) for t in src]
    dst_host = [t.cpu().numpy() for t in dst]
    per_layer_scales = scales.reshape(w.num_layers, -1)

    def mismatch(layer):
        s1 = [np.ascontiguousarray(a[layer:layer + 1]) for a in src_host]
        ref = _dst(w1, DTYPE_FP8_E4M3)
        oracle.relayout_convert(s1, ref, src_dtype=DTYPE_BF16, dst_dtype=DTYPE_FP8_E4M3,
                                per_head=1, scales=per_layer_scales[layer], **_geometry(w1))
        return not all(np.array_equal(d[layer:layer + 1], a) for a, d in zip(ref, dst_host))

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        bad = [layer for layer, m in enumerate(ex.map(mismatch, range(w.num_layers))) if m]
    assert not bad, f"layers {bad[:5]} differ from the oracle"
    per = [torch.full(w.dst_shape(), 0xFF, dtype=torch.uint8, device="cuda")
           for _ in range(w.dst_tp)]
    with RelayoutPlan(src, per, convert=conv, **w.geometry()) as plan:
        for layer in range(w.num_layers):
            plan.run_layer(layer)
        torch.cuda.synchronize()
    for a, b in zip(dst, per):
        assert torch.equal(a, b)


@pytest.mark.parametrize("seed", range(16))
def test_fuzzed_conversions(seed):
    """Random valid geometries, both directions, per-head or per-(layer, component)
    scales, random bit patterns: every launch mode equals the converting oracle."""
    from fuzz_cases import random_workload
    quant = seed % 2 == 0
    w = random_workload(seed, max_tokens=400, elem_bytes=2 if quant else 1,
                        head_dim_multiple=16)
    rng = np.random.default_rng(seed + 500)
    per_head = (seed // 2) % 2
    src_dtype, dst_dtype = (DTYPE_BF16, DTYPE_FP8_E4M3) if quant else (DTYPE_FP8_E4M3,
                                                                        DTYPE_BF16)
    scales = _scales(rng, w, per_head) if quant else _scales(rng, w, per_head, 0.5, 1e3)
    modes = ("all", "layer", "ranges") if w.num_layers > 1 else ("all", "layer")
    _check(w, _src_bits(rng, w, src_dtype), src_dtype, dst_dtype, per_head, scales, modes)
