"""GPU parity of the layout-generic relayout against the CPU oracle (bit-exact)."""
import numpy as np
import pytest

import oracle
from oracle import pd_pages
import workloads as wl
from prefill_decode_paged_gb300 import (RelayoutPlan, layout_of_views, pack_plan,
                                        unpack_plan)
from prefill_decode_paged_gb300.kv_relayout import DTYPE_BF16, DTYPE_FP8_E4M3

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    import gc
    import torch
    gc.collect()
    torch.cuda.empty_cache()


def _w(seed, **kw):
    base = dict(num_layers=3, num_components=2, kv_heads=8, head_dim=64, elem_bytes=2,
                src_tp=4, dst_tp=2, src_block=16, dst_block=64, seq_lens=[300, 1, 77, 0, 129])
    base.update(kw)
    return wl.custom("glay", seed, **base)


# a plain head split, and heads replicated on both sides (H = 2 on 4 prefill and
# 8 decode shards: read from the first prefill copy, written to all decode copies)
GEOS = {"split": {}, "replicated": dict(kv_heads=2, src_tp=4, dst_tp=8, src_block=5,
                                        dst_block=16)}


def _tables(w):
    g = w.geometry()
    keys = ("num_layers", "num_components", "kv_heads", "head_dim", "src_tp", "dst_tp",
            "src_block", "dst_block", "seq_lens", "src_off", "src_bt", "dst_off", "dst_bt")
    return {k: g[k] for k in keys}


def _np_t(a):
    import torch
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


def decode_family(w, kind, dtype=np.uint16, fill=0xFFFF):
    """numpy buffers, numpy views and the matching torch buffers/views of a decode side."""
    L, C, N, B, Hl, D = w.dst_shape()
    if kind == "standard":
        shapes, view = (L, C, N, B, Hl, D), lambda b, l, c: b[l, c]
    elif kind == "hnd":
        shapes, view = (L, C, N, Hl, B, D), lambda b, l, c: b[l, c].transpose(0, 2, 1, 3)
    elif kind == "kv_interleaved":
        shapes, view = (L, N, C, B, Hl, D), lambda b, l, c: b[l, :, c]
    else:
        raise ValueError(kind)
    bufs = [np.full(shapes, fill, dtype) for _ in range(w.dst_tp)]
    tbufs = [_np_t(b) for b in bufs]
    tview = {"standard": lambda b, l, c: b[l, c],
             "hnd": lambda b, l, c: b[l, c].permute(0, 2, 1, 3),
             "kv_interleaved": lambda b, l, c: b[l, :, c]}[kind]
    nv = [[[view(b, l, c) for c in range(C)] for l in range(L)] for b in bufs]
    tv = [[[tview(b, l, c) for c in range(C)] for l in range(L)] for b in tbufs]
    return bufs, nv, tbufs, tv


@pytest.mark.parametrize("geo", sorted(GEOS))
@pytest.mark.parametrize("kind", ["standard", "hnd", "kv_interleaved"])
@pytest.mark.parametrize("mode", ["all", "layer"])
def test_decode_layouts_match_the_oracle(kind, mode, geo):
    import torch
    w = _w(1, **GEOS[geo])
    src_np = w.src_pools_numpy()
    sv = oracle.standard_views(src_np, w.num_layers, 2, w.src_num_blocks, w.src_block,
                               wl.heads_per_shard(w.kv_heads, w.src_tp), w.head_dim)
    ref_bufs, ref_views, _, _ = decode_family(w, kind)
    oracle.relayout_general(sv, ref_views, **_tables(w))
    src = [_np_t(a) for a in src_np]
    _, _, tbufs, tviews = decode_family(w, kind)
    with RelayoutPlan(src, None, dst_layout=layout_of_views(tviews), **w.geometry()) as plan:
        if mode == "all":
            plan.run_all()
        else:
            for layer in range(w.num_layers):
                plan.run_layer(layer)
        torch.cuda.synchronize()
    for a, t in zip(ref_bufs, tbufs):
        assert np.array_equal(t.cpu().numpy().view(np.uint16), a)


def test_head_major_prefill_and_per_layer_decode_tensors():
    """Prefill pools head-major in each block; decode side one K and one V tensor per
    layer and shard (as engines that allocate per-layer caches do)."""
    import torch
    w = _w(2)
    L, C, N, B, Hl, D = w.src_shape()
    std = w.src_pools_numpy()
    hnd = [np.ascontiguousarray(a.transpose(0, 1, 2, 4, 3, 5)) for a in std]
    ths = [_np_t(a) for a in hnd]
    sv_t = [[[t[l, c].permute(0, 2, 1, 3) for c in range(C)] for l in range(L)] for t in ths]
    Ld, Cd, Nd, Bd, Hd, Dd = w.dst_shape()
    per = [[[torch.full((Nd, Bd, Hd, Dd), -1, dtype=torch.int16, device="cuda")
             for _ in range(Cd)] for _ in range(Ld)] for _ in range(w.dst_tp)]
    with RelayoutPlan(None, None, src_layout=layout_of_views(sv_t),
                      dst_layout=layout_of_views(per), **w.geometry()) as plan:
        plan.run_all()
        torch.cuda.synchronize()
    ref = w.dst_pools_numpy()
    oracle.relayout(std, ref, **w.geometry())
    for s in range(w.dst_tp):
        for l in range(Ld):
            for c in range(Cd):
                assert np.array_equal(per[s][l][c].cpu().numpy().view(np.uint16), ref[s][l, c])


@pytest.mark.parametrize("direction", ["quant", "dequant"])
def test_layouts_with_conversion(direction):
    import torch
    rng = np.random.default_rng(3)
    w = _w(4, elem_bytes=2 if direction == "quant" else 1)
    if direction == "quant":
        src_np = [rng.integers(0, 1 << 16, w.src_shape(), dtype=np.uint16) for _ in range(4)]
        kw = dict(src_dtype=DTYPE_BF16, dst_dtype=DTYPE_FP8_E4M3)
        dt, fill = np.uint8, 0xFF
    else:
        src_np = [rng.integers(0, 256, w.src_shape(), dtype=np.uint8) for _ in range(4)]
        kw = dict(src_dtype=DTYPE_FP8_E4M3, dst_dtype=DTYPE_BF16)
        dt, fill = np.uint16, 0xFFFF
    scales = rng.uniform(0.01, 2.0, w.num_layers * 2 * 8).astype(np.float32)
    sv = oracle.standard_views(src_np, w.num_layers, 2, w.src_num_blocks, w.src_block, 2,
                               w.head_dim)
    ref_bufs, ref_views, _, _ = decode_family(w, "hnd", dt, fill)
    oracle.relayout_general(sv, ref_views, per_head=1, scales=scales, **kw, **_tables(w))
    _, _, tbufs, tviews = decode_family(w, "hnd", dt, fill)
    src = [_np_t(a) for a in src_np]
    with RelayoutPlan(src, None, convert=dict(per_head=True, scales=scales, **kw),
                      dst_layout=layout_of_views(tviews), **w.geometry()) as plan:
        plan.run_all()
        torch.cuda.synchronize()
    for a, t in zip(ref_bufs, tbufs):
        assert np.array_equal(t.cpu().numpy().view(dt), a)


@pytest.mark.parametrize("geo", sorted(GEOS))
def test_pack_gives_pd_py_gather_and_unpack_gives_the_direct_relayout(geo):
    import torch
    w = _w(5, **GEOS[geo])
    src_np = w.src_pools_numpy()
    src = [_np_t(a) for a in src_np]
    total = int(w.seq_lens.sum())
    stage = torch.zeros((w.num_layers, 2, total, w.kv_heads, w.head_dim), dtype=torch.int16,
                        device="cuda")
    with pack_plan(src, stage, **w.geometry()) as plan:
        plan.run_all()
        torch.cuda.synchronize()
    got = stage.cpu().numpy().view(np.uint16)
    off = np.concatenate([[0], np.cumsum(w.seq_lens)])
    for r, n in enumerate(w.seq_lens.tolist()):
        if n == 0:
            continue
        blocks = w.src_bt[w.src_off[r]:w.src_off[r + 1]][: -(-n // w.src_block)]
        for l in range(w.num_layers):
            for c in range(2):
                want = pd_pages.gather_prefill(src_np, l, c, blocks, n, num_layers=w.num_layers,
                                               num_components=2, kv_heads=w.kv_heads,
                                               head_dim=w.head_dim, src_tp=w.src_tp,
                                               src_block=w.src_block,
                                               src_num_blocks=w.src_num_blocks)
                assert np.array_equal(got[l, c, off[r]:off[r] + n], want)
    dst = [_np_t(a) for a in w.dst_pools_numpy()]
    with unpack_plan(stage, dst, **w.geometry()) as plan:
        for layer in range(w.num_layers):
            plan.run_layer(layer)
        torch.cuda.synchronize()
    ref = w.dst_pools_numpy()
    oracle.relayout(src_np, ref, **w.geometry())
    for a, t in zip(ref, dst):
        assert np.array_equal(t.cpu().numpy().view(np.uint16), a)


def _staging_tables(w):
    """The staging buffer's documented indexing as the decode side's tables (one shard of
    one-token blocks, request r's tokens at rows sum(n[:r]) ..., block id = row)."""
    t = _tables(w)
    lens = np.asarray(w.seq_lens, dtype=np.int64)
    t.update(dst_tp=1, dst_block=1, dst_off=np.concatenate([[0], np.cumsum(lens)]),
             dst_bt=np.arange(int(lens.sum()), dtype=np.int32))
    return t


@pytest.mark.parametrize("geo", sorted(GEOS))
def test_pack_and_unpack_with_conversion(geo):
    """kv_relayout_plan_pack with a BF16 -> FP8 conversion fills the staging buffer with
    the converting oracle's gather; a bit-copy pack followed by a quantizing unpack gives
    the decode pools of one direct quantizing relayout (each element is rounded once on
    either route), bit for bit."""
    import torch
    w = _w(7, **GEOS[geo])
    rng = np.random.default_rng(17)
    src_np = [rng.integers(0, 1 << 16, w.src_shape(), dtype=np.uint16) for _ in range(w.src_tp)]
    scales = rng.uniform(0.01, 2.0, w.num_layers * 2 * w.kv_heads).astype(np.float32)
    conv = dict(src_dtype=DTYPE_BF16, dst_dtype=DTYPE_FP8_E4M3, per_head=True, scales=scales)
    src = [_np_t(a) for a in src_np]
    L, C, total = w.num_layers, 2, int(w.seq_lens.sum())
    # 1. a quantizing pack
    stage8 = torch.full((L, C, total, w.kv_heads, w.head_dim), 0xEE, dtype=torch.uint8,
                        device="cuda")
    with pack_plan(src, stage8, convert=conv, **w.geometry()) as plan:
        plan.run_all()
        torch.cuda.synchronize()
    want = np.full(tuple(stage8.shape), 0xEE, np.uint8)
    sv = oracle.standard_views(src_np, L, C, w.src_num_blocks, w.src_block,
                               max(w.kv_heads // w.src_tp, 1), w.head_dim)
    oracle.relayout_general(sv, [[[want[l, c].reshape(total, 1, w.kv_heads, w.head_dim)
                                   for c in range(C)] for l in range(L)]],
                            src_dtype=DTYPE_BF16, dst_dtype=DTYPE_FP8_E4M3, per_head=1,
                            scales=scales, **_staging_tables(w))
    assert np.array_equal(stage8.cpu().numpy(), want)
    # 2. a bit-copy pack, then a quantizing unpack into FP8 decode pools, layer by layer
    stage = torch.zeros((L, C, total, w.kv_heads, w.head_dim), dtype=torch.int16,
                        device="cuda")
    with pack_plan(src, stage, **w.geometry()) as plan:
        plan.run_all()
    dst = [torch.full(w.dst_shape(), 0xFF, dtype=torch.uint8, device="cuda")
           for _ in range(w.dst_tp)]
    with unpack_plan(stage, dst, convert=conv, **w.geometry()) as plan:
        for layer in range(L):
            plan.run_layer(layer)
        torch.cuda.synchronize()
    ref = [np.full(w.dst_shape(), 0xFF, np.uint8) for _ in range(w.dst_tp)]
    g = w.geometry()
    g.pop("elem_bytes")
    oracle.relayout_convert(src_np, ref, src_dtype=DTYPE_BF16, dst_dtype=DTYPE_FP8_E4M3,
                            per_head=1, scales=scales, **g)
    for a, t in zip(ref, dst):
        assert np.array_equal(t.cpu().numpy(), a)


@pytest.mark.parametrize("seed", range(8))
def test_fuzzed_pack_then_unpack_equals_the_direct_relayout(seed):
    """Random valid geometries (replicated heads included) through the C pack and
    unpack plans: the staging buffer holds the oracle's gather, and unpacking it gives
    the oracle's direct relayout, bit for bit (whole prompt and layer by layer)."""
    import torch
    from fuzz_cases import random_workload
    w = random_workload(seed, max_tokens=300)
    if int(w.seq_lens.sum()) == 0:
        pytest.skip("empty batch: no staging buffer")
    dt = {1: np.uint8, 2: np.uint16, 4: np.uint32}[w.elem_bytes]
    tdt = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[w.elem_bytes]
    src_np = w.src_pools_numpy()
    src = [torch.from_numpy(a.view({1: np.uint8, 2: np.int16, 4: np.int32}[w.elem_bytes])).cuda()
           for a in src_np]
    L, C, total = w.num_layers, w.num_components, int(w.seq_lens.sum())
    stage = torch.zeros((L, C, total, w.kv_heads, w.head_dim), dtype=tdt, device="cuda")
    with pack_plan(src, stage, **w.geometry()) as plan:
        plan.run_all()
        torch.cuda.synchronize()
    want = np.zeros(tuple(stage.shape), dt)
    sv = oracle.standard_views(src_np, L, C, w.src_num_blocks, w.src_block,
                               max(w.kv_heads // w.src_tp, 1), w.head_dim)
    oracle.relayout_general(sv, [[[want[l, c].reshape(total, 1, w.kv_heads, w.head_dim)
                                   for c in range(C)] for l in range(L)]],
                            **_staging_tables(w))
    assert np.array_equal(stage.cpu().numpy().view(dt), want)
    ref = w.dst_pools_numpy()
    oracle.relayout(src_np, ref, **w.geometry())
    for mode in ("all", "layer"):
        dst = [torch.from_numpy(a.view({1: np.uint8, 2: np.int16, 4: np.int32}[w.elem_bytes]))
               .cuda() for a in w.dst_pools_numpy()]
        with unpack_plan(stage, dst, **w.geometry()) as plan:
            if mode == "all":
                plan.run_all()
            else:
                for layer in range(L):
                    plan.run_layer(layer)
            torch.cuda.synchronize()
        for a, t in zip(ref, dst):
            assert np.array_equal(t.cpu().numpy().view(dt), a), mode


@pytest.mark.parametrize("geo", sorted(GEOS))
@pytest.mark.parametrize("skew", [0, 16])
@pytest.mark.parametrize("direction", ["copy", "quant", "dequant"])
@pytest.mark.parametrize("mode", ["all", "layer"])
def test_pairs_and_single_units_match_the_oracle(skew, direction, mode, geo):
    """Prefill pools on a 32-byte boundary (threads move pairs of adjacent units) and
    16 bytes past one (single units): both equal the oracle, in every conversion,
    with heads split and with heads replicated on both sides."""
    import torch
    rng = np.random.default_rng(11)
    w = _w(5, elem_bytes=1 if direction == "dequant" else 2, **GEOS[geo])
    shape = w.src_shape()
    if direction == "dequant":
        src_np = [rng.integers(0, 256, shape, dtype=np.uint8) for _ in range(w.src_tp)]
    else:
        src_np = [rng.integers(0, 1 << 16, shape, dtype=np.uint16) for _ in range(w.src_tp)]
    conv = {"copy": None,
            "quant": dict(src_dtype=DTYPE_BF16, dst_dtype=DTYPE_FP8_E4M3),
            "dequant": dict(src_dtype=DTYPE_FP8_E4M3, dst_dtype=DTYPE_BF16)}[direction]
    dt, fill = (np.uint8, 0xFF) if direction == "quant" else (np.uint16, 0xFFFF)
    scales = rng.uniform(0.01, 2.0, w.num_layers * 2 * w.kv_heads).astype(np.float32)
    sv = oracle.standard_views(src_np, w.num_layers, 2, w.src_num_blocks, w.src_block,
                               wl.heads_per_shard(w.kv_heads, w.src_tp), w.head_dim)
    ref_bufs, ref_views, _, _ = decode_family(w, "standard", dt, fill)
    extra = dict(per_head=1, scales=scales, **conv) if conv else {}
    oracle.relayout_general(sv, ref_views, **extra, **_tables(w))

    def skewed(a):
        raw = torch.empty(a.nbytes + 256, dtype=torch.uint8, device="cuda")
        t = raw[skew:skew + a.nbytes]
        t.copy_(torch.from_numpy(a.reshape(-1).view(np.uint8)).cuda())
        return t.view(torch.int16 if a.dtype == np.uint16 else torch.uint8).view(shape)

    src_t = [skewed(a) for a in src_np]
    assert all(t.data_ptr() % 32 == skew for t in src_t)
    views = [[[t[l, c] for c in range(2)] for l in range(w.num_layers)] for t in src_t]
    _, _, tbufs, _ = decode_family(w, "standard", dt, fill)
    cv = dict(per_head=True, scales=scales, **conv) if conv else None
    with RelayoutPlan(None, tbufs, src_layout=layout_of_views(views), convert=cv,
                      **w.geometry()) as plan:
        if mode == "all":
            plan.run_all()
        else:
            for l in range(w.num_layers):
                plan.run_layer(l)
        torch.cuda.synchronize()
    for ref, got in zip(ref_bufs, tbufs):
        assert np.array_equal(got.cpu().numpy().view(dt), ref)


@pytest.mark.parametrize("mode", ["all", "layer"])
def test_padded_head_stride_matches_the_oracle(mode):
    """Decode heads 144 bytes apart (rows of 128 bytes padded to a 16-byte but not a
    32-byte multiple, so the launches move one unit per access) equal the oracle."""
    import torch
    w = _w(6)
    L, C, N, B, Hl, D = w.dst_shape()
    pad = D + 8                                   # 144-byte head stride for BF16
    src_np = w.src_pools_numpy()
    sv = oracle.standard_views(src_np, w.num_layers, 2, w.src_num_blocks, w.src_block,
                               wl.heads_per_shard(w.kv_heads, w.src_tp), w.head_dim)
    ref = [np.full((L, C, N, B, Hl, pad), 0xFFFF, np.uint16) for _ in range(w.dst_tp)]
    oracle.relayout_general(sv, [[[b[l, c, ..., :D] for c in range(C)] for l in range(L)]
                                 for b in ref], **_tables(w))
    got = [torch.full((L, C, N, B, Hl, pad), -1, dtype=torch.int16, device="cuda")
           for _ in range(w.dst_tp)]
    views = [[[g[l, c, ..., :D] for c in range(C)] for l in range(L)] for g in got]
    with RelayoutPlan([_np_t(a) for a in src_np], None, dst_layout=layout_of_views(views),
                      **w.geometry()) as plan:
        if mode == "all":
            plan.run_all()
        else:
            for l in range(L):
                plan.run_layer(l)
        torch.cuda.synchronize()
    for a, g in zip(ref, got):
        assert np.array_equal(g.cpu().numpy().view(np.uint16), a)
