"""The relayout kernels with device-side address checks (a test build of the same sources).

In the checked build every row a launch computes is compared, on the GPU, with
the pool regions the plan validated before anything is read or written; a row
outside them is counted in an error word and dropped. These tests run that build
over the parity cases (head splits, odd blocks, replicated heads), every launch
mode, both conversions and every full-size workload, and require a clear error
word and the oracle's bytes. Then they narrow the checked regions so that the
check must fire: the rows it drops stay at their sentinel, every other row still
moves, and no access ever leaves the pools (a dropped row is simply not touched).
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from cases import CASES
from gpu_util import to_device, to_host
from prefill_decode_paged_gb300 import kv_relayout as kr

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def clib():
    return kr.checked_library()


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    import gc
    import torch
    gc.collect()
    torch.cuda.empty_cache()


class _Plan:
    """A plan of the checked library (raw C calls)."""

    def __init__(self, clib, w, src, dst, convert=None):
        self.lib = clib
        self.d = kr._Desc([t.data_ptr() for t in src], [t.data_ptr() for t in dst],
                          **w.geometry())
        self.h = ctypes.c_void_p()
        if convert is None:
            st = clib.kv_relayout_plan(ctypes.byref(self.d.desc), ctypes.byref(self.h))
        else:
            self.cv = kr._Convert(**convert)
            st = clib.kv_relayout_plan_convert(ctypes.byref(self.d.desc),
                                               ctypes.byref(self.cv.conv), ctypes.byref(self.h))
        assert st == 0, kr.STATUS.get(st, st)

    def run(self, mode, layers):
        lib, h = self.lib, self.h
        if mode == "all":
            assert lib.kv_relayout_all(h, None) == 0
        elif mode == "layer":
            for layer in range(layers):
                assert lib.kv_relayout_layer(h, layer, None) == 0
        else:
            # a range, then single layers passing KVR_LAUNCH_NO_WAIT after it
            first = max(1, layers // 2)
            assert lib.kv_relayout_layers(h, 0, first, None) == 0
            for layer in range(first, layers):
                assert lib.kv_relayout_layers_ex(h, layer, 1, kr.LAUNCH_NO_WAIT, None) == 0

    def status(self):
        import torch
        torch.cuda.synchronize()
        flags = ctypes.c_uint32()
        st = self.lib.kv_relayout_debug_status(self.h, ctypes.byref(flags))
        return kr.STATUS.get(st, st), flags.value

    def close(self):
        self.lib.kv_relayout_plan_destroy(self.h)


def _oracle(w, src_np):
    ref = w.dst_pools_numpy()
    oracle.relayout(src_np, ref, **w.geometry())
    return ref


@pytest.mark.parametrize("mode", ["all", "layer", "ranges"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_checked_kernels_stay_inside_the_pools(clib, case, mode):
    w = CASES[case]()
    src_np = w.src_pools_numpy()
    ref = _oracle(w, src_np)
    src = to_device(src_np, w.elem_bytes)
    dst = to_device(w.dst_pools_numpy(), w.elem_bytes)
    p = _Plan(clib, w, src, dst)
    try:
        p.run(mode, w.num_layers)
        assert p.status() == ("KVR_OK", 0)
    finally:
        p.close()
    for s, (a, b) in enumerate(zip(ref, to_host(dst, w))):
        np.testing.assert_array_equal(b, a, err_msg=f"{case} {mode} shard {s}")


@pytest.mark.parametrize("direction", ["quant", "dequant"])
def test_checked_converting_kernels(clib, direction):
    import torch
    rng = np.random.default_rng(41)
    quant = direction == "quant"
    w = wl.custom("chk_conv", 42, num_layers=3, num_components=2, kv_heads=2, head_dim=64,
                  elem_bytes=2 if quant else 1, src_tp=2, dst_tp=4, src_block=16, dst_block=5,
                  seq_lens=[130, 1, 47])
    src_np = [rng.integers(0, 1 << 16 if quant else 1 << 8, w.src_shape(),
                           dtype=np.uint16 if quant else np.uint8) for _ in range(w.src_tp)]
    src_dt, dst_dt = (kr.DTYPE_BF16, kr.DTYPE_FP8_E4M3) if quant else (kr.DTYPE_FP8_E4M3,
                                                                       kr.DTYPE_BF16)
    scales = rng.uniform(0.01, 2.0, w.num_layers * 2 * w.kv_heads).astype(np.float32)
    dnp = np.uint8 if quant else np.uint16
    ref = [np.full(w.dst_shape(), 0xFF if quant else 0xFFFF, dnp) for _ in range(w.dst_tp)]
    g = w.geometry()
    g.pop("elem_bytes")
    oracle.relayout_convert(src_np, ref, src_dtype=src_dt, dst_dtype=dst_dt, per_head=1,
                            scales=scales, **g)

    def dev(arrays):
        return [torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
                for a in arrays]
    for mode in ("all", "layer"):
        src = dev(src_np)
        dst = dev([np.full(w.dst_shape(), 0xFF if quant else 0xFFFF, dnp)
                   for _ in range(w.dst_tp)])
        p = _Plan(clib, w, src, dst, convert=dict(src_dtype=src_dt, dst_dtype=dst_dt,
                                                 scales=scales, per_head=True))
        try:
            p.run(mode, w.num_layers)
            assert p.status() == ("KVR_OK", 0)
        finally:
            p.close()
        for a, t in zip(ref, dst):
            assert np.array_equal(t.cpu().numpy().view(dnp), a)


@pytest.mark.parametrize("name", ["llama8b", "llama70b", "qwen32k_ragged", "dsv3mla",
                                  "dsv3mla_tp8"])
def test_checked_kernels_on_full_size_workloads(clib, name):
    """Every row of the whole-prompt and of every per-layer launch, checked on the GPU."""
    w = wl.get(name)
    src = w.src_pools_torch("cuda")
    dst = w.dst_pools_torch("cuda")
    p = _Plan(clib, w, src, dst)
    try:
        for mode in ("all", "layer"):
            p.run(mode, w.num_layers)
            assert p.status() == ("KVR_OK", 0), mode
    finally:
        p.close()


def test_narrowed_regions_make_the_check_fire(clib):
    """With the end of every pool region (up to one (layer, component) plane) taken out
    of the checked regions, the rows there are flagged and dropped: they keep the
    sentinel, every other row is the oracle's, and the error word clears once read."""
    w = wl.custom("chk_narrow", 43, num_layers=3, num_components=2, kv_heads=4, head_dim=32,
                  elem_bytes=2, src_tp=2, dst_tp=4, src_block=16, dst_block=32,
                  seq_lens=[200, 33])
    L, C, N, B, Hl, D = w.src_shape()
    src_plane = N * B * Hl * D * w.elem_bytes
    _, _, Nd, Bd, Hd, _ = w.dst_shape()
    dst_plane = Nd * Bd * Hd * D * w.elem_bytes
    src_np = w.src_pools_numpy()
    ref = _oracle(w, src_np)
    src = to_device(src_np, w.elem_bytes)
    dst = to_device(w.dst_pools_numpy(), w.elem_bytes)
    p = _Plan(clib, w, src, dst)
    try:
        # the smaller plane: every byte taken out lies in a last (layer, component) plane
        assert clib.kv_relayout_debug_narrow(p.h, min(src_plane, dst_plane)) == 0
        p.run("all", w.num_layers)
        name, flags = p.status()
        assert name == "KVR_ERR_DEVICE_BOUNDS" and flags != 0
        assert p.status() == ("KVR_OK", 0)          # read and cleared
    finally:
        p.close()
    got = to_host(dst, w)
    sentinel = w._sentinel_value(0xFF)
    dropped = 0
    for a, b in zip(ref, got):
        # rows outside the last (layer, component) plane are untouched by the narrowing
        keep = np.ones(a.shape[:2], bool)
        keep[L - 1, C - 1] = False
        np.testing.assert_array_equal(b[keep], a[keep])
        # inside it, a row is either the oracle's or dropped (sentinel), never wrong
        last, want = b[L - 1, C - 1], a[L - 1, C - 1]
        assert np.all((last == want) | (last == sentinel))
        dropped += int(((last == sentinel) & (want != sentinel)).sum())
    assert dropped > 0


@pytest.mark.parametrize("seed", range(32))
def test_checked_kernels_on_fuzzed_geometries(clib, seed):
    """Random valid geometries (TP splits and replication, block sizes 1-256, element
    widths, ragged and empty prompts, shared prefixes), every launch mode."""
    from fuzz_cases import random_workload
    w = random_workload(seed + 100, max_tokens=400)
    src_np = w.src_pools_numpy()
    ref = _oracle(w, src_np)
    src = to_device(src_np, w.elem_bytes)
    for mode in ("all", "layer", "ranges"):
        dst = to_device(w.dst_pools_numpy(), w.elem_bytes)
        p = _Plan(clib, w, src, dst)
        try:
            p.run(mode, w.num_layers)
            assert p.status() == ("KVR_OK", 0), mode
        finally:
            p.close()
        for s, (a, b) in enumerate(zip(ref, to_host(dst, w))):
            np.testing.assert_array_equal(b, a, err_msg=f"seed {seed} {mode} shard {s}")
