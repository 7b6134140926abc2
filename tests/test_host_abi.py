"""Host-side tests of the C ABI (no GPU): exports, validation, byte counts, and the
kernel's work decomposition walked on the CPU against the oracle."""
import ctypes
import dataclasses
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import workloads as wl
from cases import CASES
from kvcheck import check_dst, expected_from_src
from prefill_decode_paged_gb300 import build as kbuild
from prefill_decode_paged_gb300 import kv_relayout as kr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kv_relayout.h")
EMU_SRC = os.path.join(ROOT, "tests", "csrc", "kvr_emulate.cpp")
EMU_LIB = os.path.join(ROOT, "tests", "_build", "libkvr_emulate.so")
SMS = 152


@pytest.fixture(scope="session")
def cuda_lib():
    kbuild.build()
    return kr.library()


@pytest.fixture(scope="session")
def emu():
    os.makedirs(os.path.dirname(EMU_LIB), exist_ok=True)
    srcs = [EMU_SRC, os.path.join(kbuild.CSRC, "plan.cpp")]
    stale = not os.path.exists(EMU_LIB) or any(
        os.path.getmtime(f) > os.path.getmtime(EMU_LIB)
        for f in kbuild._inputs() + [EMU_SRC])
    if stale:
        subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-I", kbuild.INCLUDE,
                        "-I", kbuild.CSRC, *srcs, "-o", EMU_LIB], check=True)
    lib = ctypes.CDLL(EMU_LIB)
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.emu_relayout.restype = i64
    lib.emu_relayout.argtypes = [p, ctypes.c_int, i32, p]
    lib.emu_check.restype = i64
    lib.emu_check.argtypes = [p, ctypes.c_int, i32, p]
    lib.emu_plan_info.restype = i32
    lib.emu_plan_info.argtypes = [p, ctypes.c_int, p]
    lib.emu_fastdiv_check.restype = i64
    lib.emu_fastdiv_check.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    lib.emu_range_launch.restype = i32
    lib.emu_range_launch.argtypes = [p, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32, i32,
                                     i32, p]
    lib.emu_fastdiv_check_one.restype = i64
    lib.emu_fastdiv_check_one.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    return lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_relayout_\w+)\s*\(", text)))


def fake_pools(w, base=1 << 40, gap=1 << 20):
    """Distinct, non-overlapping, 16-B aligned device addresses (never dereferenced)."""
    src, dst, at = [], [], base
    for _ in range(w.src_tp):
        src.append(at)
        at += (w.src_pool_bytes() + gap) // 256 * 256 + 256
    for _ in range(w.dst_tp):
        dst.append(at)
        at += (w.dst_pool_bytes() + gap) // 256 * 256 + 256
    return src, dst


def status_of(fn):
    try:
        fn()
    except kr.KVRelayoutError as e:
        return e.name
    return "KVR_OK"


# -- exports ---------------------------------------------------------------------

def test_library_exports_every_declared_symbol(cuda_lib):
    names = declared_functions()
    assert set(names) == set(kr.EXPORTS)
    for n in names:
        assert hasattr(cuda_lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", kr.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kv_relayout_\w+)", out))
    assert set(names) <= exported


def test_product_library_has_no_device_checks(cuda_lib):
    """The device-side address checks exist only in the checked test build."""
    flags = ctypes.c_uint32(7)
    assert kr.STATUS[cuda_lib.kv_relayout_debug_status(None, ctypes.byref(flags))] == \
        "KVR_ERR_UNSUPPORTED"
    assert flags.value == 0
    assert kr.STATUS[cuda_lib.kv_relayout_debug_narrow(None, 0)] == "KVR_ERR_UNSUPPORTED"


def test_strerror_names_every_status(cuda_lib):
    for code in kr.STATUS:
        assert cuda_lib.kv_relayout_strerror(code)
    assert cuda_lib.kv_relayout_strerror(12345) == b"unknown status"


# -- validation (host only: kv_relayout_desc_bytes never touches the device) -----

def _geo(w, **over):
    g = w.geometry()
    g.update(over)
    return g


def test_desc_bytes_are_the_pages_kv_per_token_times_length(cuda_lib):
    for name, per_token in (("llama70b", 327680), ("qwen32k", 262144), ("dsv3mla", 70272),
                            ("llama8b", 131072)):
        w = wl.get(name)
        s, d = fake_pools(w)
        r, wr = kr.desc_bytes(s, d, **w.geometry())
        assert r == wr == per_token * int(w.seq_lens.sum())
    w = wl.llama70b()
    s, d = fake_pools(w)
    assert kr.desc_bytes(s, d, **w.geometry())[0] == 1_342_177_280


def test_every_error_is_a_status(cuda_lib):
    w = wl.custom("v", 5, num_layers=2, num_components=2, kv_heads=8, head_dim=64, elem_bytes=2,
                  src_tp=4, dst_tp=8, src_block=16, dst_block=32, seq_lens=[100, 40, 0])
    s, d = fake_pools(w)
    ok = lambda **o: (lambda: kr.desc_bytes(o.pop("src", s), o.pop("dst", d), **_geo(w, **o)))
    assert status_of(ok()) == "KVR_OK"
    # scalar ranges
    assert status_of(ok(num_layers=0)) == "KVR_ERR_INVALID_ARG"
    assert status_of(ok(num_components=3)) == "KVR_ERR_INVALID_ARG"
    assert status_of(ok(src_block=0)) == "KVR_ERR_INVALID_ARG"
    assert status_of(ok(dst_num_blocks=0)) == "KVR_ERR_INVALID_ARG"
    assert status_of(ok(elem_bytes=3)) == "KVR_ERR_UNSUPPORTED"
    assert status_of(ok(elem_bytes=8)) == "KVR_ERR_UNSUPPORTED"
    assert status_of(ok(dst_tp=3, dst=d[:3])) == "KVR_ERR_UNSUPPORTED"       # 8 % 3
    assert status_of(ok(kv_heads=32, src_tp=32)) == "KVR_ERR_UNSUPPORTED"    # > KVR_MAX_TP
    # alignment
    assert status_of(ok(head_dim=4)) == "KVR_ERR_ALIGNMENT"                  # 8-byte rows
    assert status_of(ok(src=[s[0] + 8] + s[1:])) == "KVR_ERR_ALIGNMENT"
    assert status_of(ok(dst=d[:7] + [d[7] + 4])) == "KVR_ERR_ALIGNMENT"
    # null pools
    assert status_of(ok(src=s[:3] + [0])) == "KVR_ERR_INVALID_ARG"
    # tables
    lens = w.seq_lens.copy(); lens[1] = -1
    assert status_of(ok(seq_lens=lens)) == "KVR_ERR_INVALID_ARG"
    lens = w.seq_lens.copy(); lens[0] = 200                                  # table too short
    assert status_of(ok(seq_lens=lens)) == "KVR_ERR_TABLE_SHORT"
    soff = w.src_off.copy(); soff[2] = soff[1] - 1
    assert status_of(ok(src_off=soff)) == "KVR_ERR_INVALID_ARG"
    sbt = w.src_bt.copy(); sbt[3] = w.src_num_blocks
    assert status_of(ok(src_bt=sbt)) == "KVR_ERR_BLOCK_RANGE"
    dbt = w.dst_bt.copy(); dbt[0] = -1
    assert status_of(ok(dst_bt=dbt)) == "KVR_ERR_BLOCK_RANGE"
    dbt = w.dst_bt.copy(); dbt[w.dst_off[1]] = dbt[0]                        # two requests
    assert status_of(ok(dst_bt=dbt)) == "KVR_ERR_DST_ALIAS"
    dbt = w.dst_bt.copy(); dbt[1] = dbt[0]                                   # one request
    assert status_of(ok(dst_bt=dbt)) == "KVR_ERR_DST_ALIAS"
    # pool overlaps
    assert status_of(ok(dst=[d[0]] * 8)) == "KVR_ERR_POOL_OVERLAP"
    assert status_of(ok(dst=[s[1]] + d[1:])) == "KVR_ERR_POOL_OVERLAP"
    assert status_of(ok(dst=[s[0] + 16] + d[1:])) == "KVR_ERR_POOL_OVERLAP"


def test_replicated_heads_bytes_and_refusals(cuda_lib):
    """A TP degree that is a multiple of H replicates heads: each is read once and
    written to every decode shard that holds it; a degree that neither divides nor is
    a multiple of H is refused."""
    for H, tp, copies in ((1, (1, 8), 8), (2, (8, 1), 1), (2, (4, 8), 4), (8, (8, 16), 2),
                          (1, (16, 16), 16)):
        w = wl.custom("r", 7, num_layers=3, num_components=2, kv_heads=H, head_dim=64,
                      elem_bytes=2, src_tp=tp[0], dst_tp=tp[1], src_block=16, dst_block=32,
                      seq_lens=[100, 40, 0])
        s, d = fake_pools(w)
        r, wr = kr.desc_bytes(s, d, **w.geometry())
        assert r == 140 * 3 * 2 * H * 64 * 2
        assert wr == copies * r
    w = wl.custom("r", 7, num_layers=1, num_components=2, kv_heads=2, head_dim=64,
                  elem_bytes=2, src_tp=2, dst_tp=2, src_block=16, dst_block=32, seq_lens=[5])
    s, d = fake_pools(w)
    for tp in ((3, 2), (2, 3), (5, 1), (1, 5)):                 # neither divisor nor multiple
        big_s = [s[0] + k * (1 << 24) for k in range(tp[0])]
        big_d = [d[-1] + (1 << 32) + k * (1 << 24) for k in range(tp[1])]
        assert status_of(lambda: kr.desc_bytes(big_s, big_d, **_geo(w, src_tp=tp[0],
                                                                     dst_tp=tp[1]))) \
            == "KVR_ERR_UNSUPPORTED"
    # decode copies of one head are separate pools: sharing one is an overlap
    w = wl.custom("r", 7, num_layers=1, num_components=1, kv_heads=1, head_dim=64,
                  elem_bytes=2, src_tp=1, dst_tp=4, src_block=16, dst_block=16, seq_lens=[5])
    s, d = fake_pools(w)
    assert status_of(lambda: kr.desc_bytes(s, [d[0], d[1], d[1], d[3]], **w.geometry())) \
        == "KVR_ERR_POOL_OVERLAP"


def test_permitted_edge_cases(cuda_lib):
    w = wl.custom("e", 6, num_layers=2, num_components=2, kv_heads=8, head_dim=64, elem_bytes=2,
                  src_tp=4, dst_tp=8, src_block=16, dst_block=32, seq_lens=[96, 40, 0])
    s, d = fake_pools(w)
    # reserved-but-unused decode entries may be anything, prefill ids may repeat
    assert w.dst_off[1] == 4 and w.dst_off[3] - w.dst_off[2] == 1
    dbt = w.dst_bt.copy()
    dbt[w.dst_off[1] - 1] = 10 ** 6          # request 0: the block reserved for token 97
    dbt[w.dst_off[3] - 1] = dbt[0]           # request 2 (empty prompt): its reserved block
    assert status_of(lambda: kr.desc_bytes(s, d, **_geo(w, dst_bt=dbt))) == "KVR_OK"
    sbt = w.src_bt.copy(); sbt[w.src_off[1]] = sbt[0]
    assert status_of(lambda: kr.desc_bytes(s, d, **_geo(w, src_bt=sbt))) == "KVR_OK"
    # prefill pools may overlap each other (read only)
    assert status_of(lambda: kr.desc_bytes([s[0]] * 4, d, **w.geometry())) == "KVR_OK"
    # empty batch and all-zero lengths
    e = dict(w.geometry(), seq_lens=[], src_off=[0], src_bt=[], dst_off=[0], dst_bt=[])
    assert kr.desc_bytes(s, d, **e) == (0, 0)
    z = dict(w.geometry(), seq_lens=[0, 0], src_off=[0, 0, 0], src_bt=[], dst_off=[0, 0, 0],
             dst_bt=[])
    assert kr.desc_bytes(s, d, **z) == (0, 0)


def test_plan_without_a_gpu_fails_loudly(cuda_lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    w = wl.tiny()
    s, d = fake_pools(w)
    with pytest.raises(kr.KVRelayoutError) as e:
        kr.RelayoutPlan(s, d, **w.geometry())
    assert e.value.name == "KVR_ERR_CUDA"


# -- the kernel's decomposition, walked on the CPU ----------------------------------

def _host_desc(w, src, dst):
    return kr._Desc([a.ctypes.data for a in src], [a.ctypes.data for a in dst], **w.geometry())


def _emu_run(emu, w, src, dst, layer=-1, sms=SMS):
    d = _host_desc(w, src, dst)
    n = ctypes.c_int64()
    bad = emu.emu_relayout(ctypes.byref(d.desc), sms, layer, ctypes.byref(n))
    assert bad == 0, f"{bad} chunk addresses out of bounds or misaligned"
    return n.value


def _aligned(shape, dtype, align=256, skew=0):
    """Host array whose data starts `skew` bytes past an `align`-byte boundary (the
    CUDA allocator's pools start on 256-byte boundaries)."""
    nbytes = int(np.prod(shape)) * np.dtype(dtype).itemsize
    raw = np.empty(nbytes + align + skew, dtype=np.uint8)
    off = (-raw.ctypes.data) % align + skew
    return raw[off:off + nbytes].view(dtype).reshape(shape)


def _pools(w, filled, skew=0):
    out = []
    for a in filled:
        b = _aligned(a.shape, a.dtype, skew=skew)
        b[...] = a
        out.append(b)
    return out


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("sms", [1, SMS])
def test_emulated_kernel_matches_oracle(emu, case, sms):
    w = CASES[case]()
    src = _pools(w, w.src_pools_numpy())
    ref = w.dst_pools_numpy()
    oracle.relayout(src, ref, **w.geometry())
    whole = _pools(w, w.dst_pools_numpy())
    n = _emu_run(emu, w, src, whole, sms=sms)
    # one unit per 16 bytes written: each decode copy of a replicated head is written
    copies = max(1, w.dst_tp // w.kv_heads)
    assert n * 16 == copies * oracle.transfer_bytes(w.num_layers, w.num_components,
                                                    w.kv_heads, w.head_dim, w.elem_bytes,
                                                    w.seq_lens)
    for a, b in zip(ref, whole):
        np.testing.assert_array_equal(a, b)
    per = _pools(w, w.dst_pools_numpy())
    for l in range(w.num_layers):
        assert _emu_run(emu, w, src, per, layer=l, sms=sms) * w.num_layers == n
    for a, b in zip(ref, per):
        np.testing.assert_array_equal(a, b)
    check_dst(w, whole, expected_from_src(w, src), w._sentinel_value(0xFF))


@pytest.mark.parametrize("name", ["llama8b", "llama70b", "qwen32k", "qwen32k_ragged",
                                  "dsv3mla", "dsv3mla_tp8"])
def test_full_size_launches_stay_in_bounds(emu, name):
    """Every address of the full-size launches, against the full pool extents.

    The whole-prompt launch is walked in full for the 70B workload; for the
    others the per-layer launches of the first and last layer are walked (the
    layer only adds a plane offset, so these bound every layer), plus the
    whole-prompt launch of a two-layer copy of the same batch.
    """
    w = wl.get(name)
    s, d = fake_pools(w)
    desc = kr._Desc(s, d, **w.geometry())
    # units are 16 bytes written: every decode copy of a replicated head counts
    per_layer = (w.seq_lens.sum() * w.num_components * w.kv_heads * w.head_dim * w.elem_bytes
                 * max(1, w.dst_tp // w.kv_heads))
    n = ctypes.c_int64()
    layers = [-1, 0, w.num_layers - 1] if name == "llama70b" else [0, w.num_layers - 1]
    for l in layers:
        assert emu.emu_check(ctypes.byref(desc.desc), SMS, l, ctypes.byref(n)) == 0
        assert n.value * 16 == (per_layer * (w.num_layers if l < 0 else 1))
    w2 = w.with_layers(2)
    s2, d2 = fake_pools(w2)
    desc2 = kr._Desc(s2, d2, **w2.geometry())
    assert emu.emu_check(ctypes.byref(desc2.desc), SMS, -1, ctypes.byref(n)) == 0
    assert n.value * 16 == per_layer * 2


def test_fast_division_matches_hardware_division(emu):
    assert emu.emu_fastdiv_check(4096, 1 << 22) == 0
    for d in (4097, 12345, 65535, 65536, 65537, 1 << 20, (1 << 20) + 1, 3 << 28,
              (1 << 30) + 3, (1 << 31) - 1):
        assert emu.emu_fastdiv_check_one(d, 1 << 16) == 0, d


def test_launch_shapes(emu):
    """Per-layer launches are sliced to fill the GPU; whole-prompt launches are not."""
    info = (ctypes.c_int64 * 6)()
    for name, n_items in (("llama70b", 128), ("qwen32k", 2048)):
        w = wl.get(name)
        s, d = fake_pools(w)
        desc = kr._Desc(s, d, **w.geometry())
        assert emu.emu_plan_info(ctypes.byref(desc.desc), SMS, info) == 0
        assert info[0] == n_items
        assert info[4] >= SMS                      # a per-layer launch covers every SM
        assert info[3] == n_items * w.num_layers * info[1]
        assert info[5] == w.dst_block                 # 128 KB+ decode blocks: one per tile
    # small decode blocks are grouped: MLA's 16-token (18 KB) blocks, 3 per tile (54 KB)
    w = wl.get("dsv3mla")
    s, d = fake_pools(w)
    desc = kr._Desc(s, d, **w.geometry())
    assert emu.emu_plan_info(ctypes.byref(desc.desc), SMS, info) == 0
    assert info[5] == 48
    assert info[0] == sum(-(-int(n) // 48) for n in w.seq_lens)


def test_launch_modes_and_grids_per_stream(emu):
    """Which kernel instance a kv_relayout_layers() launch runs, and its grid: an ordered
    launch whose tasks fit one wave of the prefetching instance on the stream's SMs runs
    it with a grid inside that wave; no-wait launches never prefetch; a stream with
    fewer SMs gets a grid shaped for them; long ranges run the whole-prompt instance."""
    WHOLE, LAYER, PREFETCH = 0, 1, 2
    ALL = 0xFFFFFFFF
    out = (ctypes.c_int64 * 5)()

    def shape(name, count, stream_sms=0, no_wait=False, res=4, res_pf=4):
        w = wl.get(name)
        s, d = fake_pools(w)
        desc = kr._Desc(s, d, **w.geometry())
        assert emu.emu_range_launch(ctypes.byref(desc.desc), SMS, res, res_pf, count,
                                    stream_sms, int(no_wait), out) == 0
        return out[0], out[1], out[2], out[3]

    def prefetching(name, count, stream_sms=0, no_wait=False):
        shape(name, count, stream_sms, no_wait)
        return out[4]

    # 70B: 128 items per layer
    sl, mode, grid, items = shape("llama70b", 1)
    assert items == 128 and mode == PREFETCH and grid == 512 and grid <= SMS * 4
    sl, mode, grid, _ = shape("llama70b", 1, no_wait=True)
    assert mode == LAYER and grid <= SMS * 4
    for sms in (8, 16, 32, 64, 96):
        sl, mode, grid, _ = shape("llama70b", 1, stream_sms=sms)
        if 128 < sms * 4:                     # fits one wave of the prefetching instance
            assert mode == PREFETCH and sms * 4 - 128 < grid <= sms * 4
        else:                                 # about three waves of the per-layer one
            assert mode == LAYER and grid >= 128
    # a prefetching instance with fewer resident CTAs gets its own shape
    sl, mode, grid, _ = shape("llama70b", 1, res=6, res_pf=4)
    assert mode == PREFETCH and grid <= SMS * 4
    # no residency known for the prefetching instance: never prefetch
    assert shape("llama70b", 1, res_pf=0)[1] == LAYER
    # ranges: two and four 70B layers fill most of one wave, eight do not fit it;
    # three (384 one-item CTAs on 608 slots) would leave too much of it idle
    for count in (2, 4):
        sl, mode, grid, _ = shape("llama70b", count)
        assert mode == PREFETCH and 3 * SMS < grid <= SMS * 4, count
    assert shape("llama70b", 3)[1] == WHOLE
    assert shape("llama70b", 8)[1] == WHOLE
    # which CTAs of an ordered launch prefetch: the first 5/8 of a single 70B
    # layer on the whole device; every CTA on a green-context stream, in a range
    # of layers and in a no-wait launch (whose instance does not prefetch)
    assert prefetching("llama70b", 1) == 512 * 5 // 8
    assert prefetching("llama70b", 1, stream_sms=96) == ALL
    assert prefetching("llama70b", 1, stream_sms=SMS) == 512 * 5 // 8
    assert prefetching("llama70b", 2) == ALL
    assert prefetching("llama70b", 1, no_wait=True) == ALL
    # Qwen 32K layers hold 2048 items: several waves, no prefetch
    sl, mode, grid, items = shape("qwen32k", 1)
    assert items == 2048 and mode == LAYER and grid >= SMS * 4


# -- converting relayout (host side) -------------------------------------------------

BF16, E4M3 = kr.DTYPE_BF16, kr.DTYPE_FP8_E4M3


def _conv(w, src_dtype=BF16, dst_dtype=E4M3, per_head=False, value=0.05):
    n = w.num_layers * w.num_components * (w.kv_heads if per_head else 1)
    return dict(src_dtype=src_dtype, dst_dtype=dst_dtype, per_head=per_head,
                scales=np.full(n, value, np.float32))


def test_convert_bytes_and_errors(cuda_lib):
    w = wl.llama70b()
    s, d = fake_pools(w)
    assert kr.desc_bytes(s, d, convert=_conv(w), **w.geometry()) == (1_342_177_280,
                                                                      671_088_640)
    w1 = dataclasses.replace(w, elem_bytes=1)
    assert kr.desc_bytes(s, d, convert=_conv(w1, E4M3, BF16, True), **w1.geometry()) == (
        671_088_640, 1_342_177_280)

    def st(conv, geo=None):
        return status_of(lambda: kr.desc_bytes(s, d, convert=conv, **(geo or w.geometry())))
    assert st(_conv(w, BF16, BF16)) == "KVR_ERR_UNSUPPORTED"
    assert st(_conv(w, E4M3, E4M3)) == "KVR_ERR_UNSUPPORTED"
    assert st(_conv(w, 7, E4M3)) == "KVR_ERR_UNSUPPORTED"
    assert st(_conv(w1, BF16, E4M3), w1.geometry()) == "KVR_ERR_INVALID_ARG"  # es must be 2
    assert st(_conv(w, E4M3, BF16)) == "KVR_ERR_INVALID_ARG"                  # es must be 1
    c = _conv(w); c["per_head"] = 2
    assert st(c) == "KVR_ERR_INVALID_ARG"
    for bad in (0.0, -1.0, np.inf, np.nan):
        c = _conv(w); c["scales"] = c["scales"].copy(); c["scales"][7] = bad
        assert st(c) == "KVR_ERR_INVALID_ARG", bad
    c = _conv(w); c["scales"] = np.zeros(0, np.float32)
    assert st(c) == "KVR_ERR_INVALID_ARG"
    g = dict(w.geometry(), head_dim=8)               # 16-byte BF16 rows, 8-byte FP8 rows
    assert st(_conv(w), g) == "KVR_ERR_ALIGNMENT"


@pytest.mark.parametrize("name,direction", [("llama70b", "quant"), ("llama70b", "dequant"),
                                            ("qwen32k", "quant"), ("dsv3mla", "quant"),
                                            ("dsv3mla", "dequant"), ("llama8b", "dequant")])
def test_convert_launches_stay_in_bounds(emu, name, direction):
    """Every address of the converting launches (units of 16 elements: 32 bytes on the
    BF16 side, 16 on the FP8 side) against the pools' full extents."""
    emu.emu_check_convert.restype = ctypes.c_int64
    emu.emu_check_convert.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                      ctypes.c_int32, ctypes.c_void_p]
    w = wl.get(name)
    if direction == "dequant":
        w = dataclasses.replace(w, elem_bytes=1)
        conv = _conv(w, E4M3, BF16, per_head=True)
    else:
        conv = _conv(w)
    s, d = fake_pools(w, gap=1 << 33)                 # room for 2-byte decode elements
    desc = kr._Desc(s, d, **w.geometry())
    cv = kr._Convert(**conv)
    n = ctypes.c_int64()
    units_per_layer = int(w.seq_lens.sum()) * w.num_components * w.kv_heads * w.head_dim // 16
    layers = [-1, 0, w.num_layers - 1] if name == "llama70b" else [0, w.num_layers - 1]
    for l in layers:
        assert emu.emu_check_convert(ctypes.byref(desc.desc), ctypes.byref(cv.conv), SMS, l,
                                     ctypes.byref(n)) == 0
        assert n.value == units_per_layer * (w.num_layers if l < 0 else 1)


def test_sm_stream_rejects_bad_counts_and_needs_a_gpu(cuda_lib):
    import torch
    with pytest.raises(kr.KVRelayoutError) as e:
        kr.SmStream(0)
    assert e.value.name == "KVR_ERR_INVALID_ARG"
    if not torch.cuda.is_available():
        with pytest.raises(kr.KVRelayoutError) as e:
            kr.SmStream(8)
        assert e.value.name == "KVR_ERR_CUDA"


def test_geometry_past_the_kernels_32_bit_indices_is_unsupported(cuda_lib):
    """Row sizes, tile sizes and work-list lengths the kernel indexes in 32 bits are
    refused at plan time with a status, not truncated."""
    def st(**geo):
        w = wl.custom("big", 11, **geo)
        s, d = fake_pools(w)
        return status_of(lambda: kr.desc_bytes(s, d, **w.geometry()))
    base = dict(num_layers=2, num_components=2, kv_heads=8, head_dim=128, elem_bytes=2,
                src_tp=1, dst_tp=1, src_block=16, dst_block=32, seq_lens=[40])
    assert st(**base) == "KVR_OK"
    # one row of 2^31 bytes
    assert st(**dict(base, head_dim=1 << 30)) == "KVR_ERR_UNSUPPORTED"
    # one decode block of Bd * C * H rows of 16 units each: 2^24 * 2 * 8 * 16 = 2^32 units
    assert st(**dict(base, dst_block=1 << 24)) == "KVR_ERR_UNSUPPORTED"
    # the largest decode block whose units still fit: 2^22 * 256 = 2^30 units
    assert st(**dict(base, dst_block=1 << 22)) == "KVR_OK"


def _emu_range(emu, w, src, dst, first, count, copy=1, sms=SMS):
    emu.emu_relayout_range.restype = ctypes.c_int64
    emu.emu_relayout_range.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
    d = _host_desc(w, src, dst) if copy else kr._Desc(src, dst, **w.geometry())
    n = ctypes.c_int64()
    bad = emu.emu_relayout_range(ctypes.byref(d.desc), sms, first, count, copy, ctypes.byref(n))
    return bad, n.value


@pytest.mark.parametrize("groups", [[5], [1, 1, 1, 1, 1], [2, 3], [3, 2], [1, 3, 1]])
def test_emulated_layer_ranges_match_the_oracle(emu, groups):
    """Any split of the layers into ranges, one launch per range, gives the oracle's
    result; each launch visits exactly its layers' units."""
    w = wl.custom("rng", 31, num_layers=5, num_components=2, kv_heads=8, head_dim=64,
                  elem_bytes=2, src_tp=4, dst_tp=2, src_block=16, dst_block=64,
                  seq_lens=[300, 1, 77, 0, 129])
    src = _pools(w, w.src_pools_numpy())
    ref = w.dst_pools_numpy()
    oracle.relayout(src, ref, **w.geometry())
    dst = _pools(w, w.dst_pools_numpy())
    per_layer_units = int(w.seq_lens.sum()) * 2 * 8 * 64 * 2 // 16
    first = 0
    for count in groups:
        bad, n = _emu_range(emu, w, src, dst, first, count)
        assert bad == 0 and n == count * per_layer_units
        first += count
    for a, b in zip(ref, dst):
        np.testing.assert_array_equal(a, b)
    check_dst(w, dst, expected_from_src(w, src), w._sentinel_value(0xFF))


def test_full_size_layer_ranges_stay_in_bounds(emu):
    w = wl.get("llama70b")
    s, d = fake_pools(w)
    per_layer_units = 4096 * 2 * 8 * 128 * 2 // 16
    for first, count in ((0, 8), (72, 8), (0, 80), (40, 2), (79, 1)):
        bad, n = _emu_range(emu, w, s, d, first, count, copy=0)
        assert bad == 0 and n == count * per_layer_units, (first, count)
    for first, count in ((-1, 2), (79, 2), (0, 81)):
        bad, _ = _emu_range(emu, w, s, d, first, count, copy=0)
        assert bad == kr.KVRelayoutError(-7, "").status


@pytest.mark.parametrize("seed", range(60))
def test_fuzzed_geometries_on_the_emulated_kernel(emu, seed):
    """Random valid geometries: every launch mode of the kernel's decomposition, walked
    on the CPU with bounds checks, equals the oracle."""
    from fuzz_cases import random_workload
    w = random_workload(seed)
    # every fourth seed: prefill pools 16 bytes past a 32-byte boundary (rows
    # taken one unit per access instead of in pairs)
    src = _pools(w, w.src_pools_numpy(), skew=16 if seed % 4 == 3 else 0)
    ref = w.dst_pools_numpy()
    oracle.relayout(src, ref, **w.geometry())
    sms = [1, 7, SMS][seed % 3]
    whole = _pools(w, w.dst_pools_numpy())
    _emu_run(emu, w, src, whole, sms=sms)
    for a, b in zip(ref, whole):
        np.testing.assert_array_equal(a, b)
    per = _pools(w, w.dst_pools_numpy())
    for l in range(w.num_layers):
        _emu_run(emu, w, src, per, layer=l, sms=sms)
    for a, b in zip(ref, per):
        np.testing.assert_array_equal(a, b)
    if w.num_layers > 1:
        rng_ = _pools(w, w.dst_pools_numpy())
        bad, _ = _emu_range(emu, w, src, rng_, 0, w.num_layers - 1, sms=sms)
        assert bad == 0
        bad, _ = _emu_range(emu, w, src, rng_, w.num_layers - 1, 1, sms=sms)
        assert bad == 0
        for a, b in zip(ref, rng_):
            np.testing.assert_array_equal(a, b)


def _pairs(emu, w, src, dst, convert=None):
    d = kr._Desc(src, dst, **w.geometry())
    cv = kr._Convert(**convert) if convert else None
    return emu.emu_plan_pairs(ctypes.byref(d.desc), None, None,
                              ctypes.byref(cv.conv) if cv else None)


def test_pairs_of_units_only_where_every_row_allows_them(emu):
    """Threads move pairs of adjacent units (32-byte accesses) exactly when rows hold
    an even number of units and every row of both sides (every decode copy of a
    replicated head too) starts on a 32-byte boundary."""
    emu.emu_plan_pairs.restype = ctypes.c_int32
    emu.emu_plan_pairs.argtypes = [ctypes.c_void_p] * 4

    def case(**kw):
        base = dict(num_layers=2, num_components=2, kv_heads=8, head_dim=128, elem_bytes=2,
                    src_tp=4, dst_tp=8, src_block=16, dst_block=32, seq_lens=[40, 7])
        base.update(kw)
        return wl.custom("pairs", 0, **base)

    w = case()
    s, d = fake_pools(w)
    assert _pairs(emu, w, s, d) == 1                              # 16 units a row
    assert _pairs(emu, w, s[:1] + [s[1] + 16] + s[2:], d) == 0    # one shard 16 B off
    assert _pairs(emu, w, s, d[:-1] + [d[-1] + 32]) == 1          # 32 B off is fine
    w = case(head_dim=8)                                          # one unit a row
    assert _pairs(emu, w, *fake_pools(w)) == 0
    w = case(head_dim=24)                                         # three units, odd
    assert _pairs(emu, w, *fake_pools(w)) == 0
    w = case(head_dim=16, elem_bytes=1)                           # 16 B rows: one unit
    assert _pairs(emu, w, *fake_pools(w)) == 0
    w = case(kv_heads=2, src_tp=4)                                # replicated heads
    s, d = fake_pools(w)
    assert _pairs(emu, w, s, d) == 1
    assert _pairs(emu, w, s, d[:3] + [d[3] + 16] + d[4:]) == 0    # one decode copy off
    # conversions: a unit is 16 elements (32 BF16 bytes, 16 FP8 bytes)
    w = case(head_dim=32)
    q = dict(src_dtype=1, dst_dtype=2, scales=np.ones(2 * 2, np.float32))
    assert _pairs(emu, w, *fake_pools(w), convert=q) == 1
    w = case(head_dim=16)
    assert _pairs(emu, w, *fake_pools(w), convert=q) == 0
    # rows of 32 bytes (two units) 48 bytes apart on the decode side: not aligned
    w = case(head_dim=16)
    s, d = fake_pools(w)
    L, C, N, B, Hl, D = w.dst_shape()
    for pad, want in ((24, 0), (32, 1)):
        bufs = [_aligned((L, C, N, B, Hl, pad), np.uint16) for _ in range(w.dst_tp)]
        lay = kr._Layout(**kr.layout_of_views(
            [[[b[l, c, ..., :D] for c in range(C)] for l in range(L)] for b in bufs]))
        dd = kr._Desc(s, d, **w.geometry())
        assert emu.emu_plan_pairs(ctypes.byref(dd.desc), None, ctypes.byref(lay.layout),
                                  None) == want, pad


ABI_CLIENT_SRC = os.path.join(ROOT, "tests", "csrc", "abi_client.c")
ABI_CLIENT = os.path.join(ROOT, "tests", "_build", "abi_client")


def build_abi_client():
    """gcc -std=c99 against the C header alone, linked to the library and the oracle."""
    kbuild.build()
    oracle.build()
    cuda = os.path.dirname(os.path.dirname(kbuild.nvcc_path()))
    lib_dir = os.path.dirname(kr.LIB_PATH)
    ora = oracle.build()
    os.makedirs(os.path.dirname(ABI_CLIENT), exist_ok=True)
    cuda_lib = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.isdir(d))
    # the header on its own is strict ISO C99 (the CUDA runtime header the client
    # also includes is not, so the client itself is built without -pedantic)
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-fsyntax-only", "-x", "c", "-I", kbuild.INCLUDE, "-"],
                   input='#include "kv_relayout.h"\n', text=True, check=True)
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror",
           "-I", kbuild.INCLUDE, "-I", os.path.join(cuda, "include"), ABI_CLIENT_SRC,
           kr.LIB_PATH, ora, "-L", cuda_lib, "-lcudart",
           f"-Wl,-rpath,{lib_dir}:{os.path.dirname(ora)}:{cuda_lib}", "-o", ABI_CLIENT]
    subprocess.run(cmd, check=True)
    return ABI_CLIENT


def test_plain_c_client_validates_on_the_host():
    """A C99 program that includes only kv_relayout.h: byte counts and the documented
    error statuses, on fake pool addresses (no GPU call)."""
    exe = build_abi_client()
    out = subprocess.run([exe, "host"], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "host: ok" in out.stdout


# -- pack / unpack through a staging buffer ---------------------------------------------

def test_staging_bytes_and_pack_unpack_statuses(cuda_lib):
    """kv_relayout_staging_bytes is L * C * (sum of n) * H * D * element bytes (host
    only); pack and unpack plans refuse what they cannot describe before any CUDA call,
    and otherwise need the GPU."""
    import ctypes
    import torch
    w = wl.llama70b()
    g = w.geometry()
    assert kr.staging_bytes(2, **g) == 4096 * 80 * 2 * 8 * 128 * 2 == 1_342_177_280
    assert kr.staging_bytes(1, **g) == 671_088_640
    q = wl.qwen32k()
    assert kr.staging_bytes(2, **q.geometry()) == 4 * 32768 * 262_144      # 256 KB per token
    assert status_of(lambda: kr.staging_bytes(3, **g)) == "KVR_ERR_INVALID_ARG"
    assert status_of(lambda: kr.staging_bytes(2, **dict(g, seq_lens=[-1], src_off=[0, 0],
                                                        dst_off=[0, 0]))) == \
        "KVR_ERR_INVALID_ARG"
    s, _ = fake_pools(w)
    lib = kr.library()

    def plan(fn, desc, staging):
        h = ctypes.c_void_p(12345)
        st = fn(ctypes.byref(desc.desc), staging, None, ctypes.byref(h))
        assert h.value is None                     # *out is NULL on every failure
        return kr.STATUS[st]
    d = kr._Desc(s, None, **g)
    assert plan(lib.kv_relayout_plan_pack, d, None) == "KVR_ERR_INVALID_ARG"
    assert plan(lib.kv_relayout_plan_unpack, kr._Desc(None, None, **g), None) == \
        "KVR_ERR_INVALID_ARG"
    empty = kr._Desc(s, None, **dict(g, seq_lens=[0], src_off=[0, 0], dst_off=[0, 0]))
    assert plan(lib.kv_relayout_plan_pack, empty, 1 << 45) == "KVR_ERR_INVALID_ARG"
    if not torch.cuda.is_available():
        assert plan(lib.kv_relayout_plan_pack, d, 1 << 45) == "KVR_ERR_CUDA"
