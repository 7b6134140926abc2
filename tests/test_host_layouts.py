"""Layouts on the host: validation of kvr_layout and the kernel's decomposition walked
on the CPU over every layout family, against the layout-generic oracle."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from prefill_decode_paged_gb300 import kv_relayout as kr
from test_host_abi import SMS, _aligned, emu, fake_pools, status_of  # noqa: F401

L_, C_ = 3, 2


def _w(seed, **kw):
    base = dict(num_layers=L_, num_components=C_, kv_heads=8, head_dim=16, elem_bytes=2,
                src_tp=4, dst_tp=2, src_block=16, dst_block=64, seq_lens=[300, 1, 77, 0])
    base.update(kw)
    return wl.custom("lay", seed, **base)


# a plain head split, and heads replicated on both sides (H = 2 on 4 prefill and
# 8 decode shards: read from the first prefill copy, written to all decode copies)
GEOS = {"split": {}, "replicated": dict(kv_heads=2, src_tp=4, dst_tp=8, src_block=5,
                                        dst_block=16)}


def _std(w, pools, side):
    if side == "src":
        return oracle.standard_views(pools, w.num_layers, w.num_components, w.src_num_blocks,
                                     w.src_block, wl.heads_per_shard(w.kv_heads, w.src_tp),
                                     w.head_dim)
    return oracle.standard_views(pools, w.num_layers, w.num_components, w.dst_num_blocks,
                                 w.dst_block, wl.heads_per_shard(w.kv_heads, w.dst_tp),
                                 w.head_dim)


def _alloc(shape, fill):
    a = _aligned(shape, np.uint16)
    a[...] = fill
    return a


def dst_family(w, kind):
    """(buffers, views[shard][layer][comp]) of a decode side in layout `kind`."""
    L, C, N, B, Hl, D = w.dst_shape()
    if kind == "standard":
        bufs = [_alloc(w.dst_shape(), 0xFFFF) for _ in range(w.dst_tp)]
        return bufs, _std(w, bufs, "dst")
    if kind == "hnd":
        bufs = [_alloc((L, C, N, Hl, B, D), 0xFFFF) for _ in range(w.dst_tp)]
        return bufs, [[[b[l, c].transpose(0, 2, 1, 3) for c in range(C)] for l in range(L)]
                      for b in bufs]
    if kind == "kv_interleaved":
        bufs = [_alloc((L, N, C, B, Hl, D), 0xFFFF) for _ in range(w.dst_tp)]
        return bufs, [[[b[l, :, c] for c in range(C)] for l in range(L)] for b in bufs]
    if kind == "separate":
        views = [[[_alloc((N, B, Hl, D), 0xFFFF) for _ in range(C)] for _ in range(L)]
                 for _ in range(w.dst_tp)]
        return [v for s in views for l in s for v in l], views
    raise ValueError(kind)


def _ranges(bufs):
    out = []
    for b in bufs:
        out += [b.ctypes.data, b.ctypes.data + b.nbytes]
    return np.array(out, dtype=np.uint64)


def _walk(emu, w, src_views, src_bufs, dst_views, dst_bufs, layer=-1, geometry=None,
          copy=1):
    emu.emu_walk_ex.restype = ctypes.c_int64
    emu.emu_walk_ex.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64, ctypes.c_void_p,
                                                        ctypes.c_int64, ctypes.c_int,
                                                        ctypes.c_int32, ctypes.c_int32,
                                                        ctypes.c_void_p]
    g = geometry or w.geometry()
    d = kr._Desc(None, None, **g)
    sl = kr._Layout(**kr.layout_of_views(src_views))
    dl = kr._Layout(**kr.layout_of_views(dst_views))
    sr, dr = _ranges(src_bufs), _ranges(dst_bufs)
    n = ctypes.c_int64()
    bad = emu.emu_walk_ex(ctypes.byref(d.desc), ctypes.byref(sl.layout), ctypes.byref(dl.layout),
                          None, sr.ctypes.data, len(src_bufs), dr.ctypes.data, len(dst_bufs),
                          SMS, layer, copy, ctypes.byref(n))
    assert bad == 0, f"{bad} rows or units outside their buffers / misaligned"
    return n.value


def _tables(g):
    keys = ("num_layers", "num_components", "kv_heads", "head_dim", "src_tp", "dst_tp",
            "src_block", "dst_block", "seq_lens", "src_off", "src_bt", "dst_off", "dst_bt")
    return {k: g[k] for k in keys}


@pytest.mark.parametrize("geo", sorted(GEOS))
@pytest.mark.parametrize("kind", ["standard", "hnd", "kv_interleaved", "separate"])
@pytest.mark.parametrize("mode", ["all", "layer"])
def test_emulated_kernel_on_decode_layouts(emu, kind, mode, geo):
    w = _w(1, **GEOS[geo])
    src_bufs = [_aligned(w.src_shape(), np.uint16) for _ in range(w.src_tp)]
    for a, b in zip(src_bufs, w.src_pools_numpy()):
        a[...] = b
    sv = _std(w, src_bufs, "src")
    ref_bufs, ref_views = dst_family(w, kind)
    oracle.relayout_general(sv, ref_views, **_tables(w.geometry()))
    got_bufs, got_views = dst_family(w, kind)
    layers = [-1] if mode == "all" else range(w.num_layers)
    for l in layers:
        _walk(emu, w, sv, src_bufs, got_views, got_bufs, layer=l)
    for a, b in zip(ref_bufs, got_bufs):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("geo", sorted(GEOS))
def test_emulated_kernel_head_major_prefill(emu, geo):
    w = _w(2, **GEOS[geo])
    std_src = w.src_pools_numpy()
    L, C, N, B, Hl, D = w.src_shape()
    hnd = []
    for s in std_src:
        a = _aligned((L, C, N, Hl, B, D), np.uint16)
        a[...] = s.transpose(0, 1, 2, 4, 3, 5)
        hnd.append(a)
    sv = [[[b[l, c].transpose(0, 2, 1, 3) for c in range(C)] for l in range(L)] for b in hnd]
    ref = w.dst_pools_numpy()
    oracle.relayout(std_src, ref, **w.geometry())
    got_bufs, got_views = dst_family(w, "standard")
    _walk(emu, w, sv, hnd, got_views, got_bufs)
    for a, b in zip(ref, got_bufs):
        np.testing.assert_array_equal(a, b)


def _staging_tables(g, side):
    """The staging buffer's documented indexing as one side's tables: one-token blocks,
    request r's tokens at rows sum(n[:r]) .. sum(n[:r + 1]) - 1 (block id = row)."""
    lens = np.asarray(g["seq_lens"], dtype=np.int64)
    total = int(lens.sum())
    t = dict(g)
    t.update({f"{side}_tp": 1, f"{side}_block": 1,
              f"{side}_off": np.concatenate([[0], np.cumsum(lens)]).astype(np.int64),
              f"{side}_bt": np.arange(total, dtype=np.int32)})
    return t


def _emu_staging(emu, w, stage, pack, pools):
    emu.emu_staging.restype = ctypes.c_int64
    emu.emu_staging.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                ctypes.c_int64, ctypes.c_int, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_void_p]
    d = kr._Desc(pools if pack else None, None if pack else pools, **w.geometry())
    sr, dr = (_ranges(pools), _ranges([stage])) if pack else (_ranges([stage]), _ranges(pools))
    n = ctypes.c_int64()
    bad = emu.emu_staging(ctypes.byref(d.desc), stage.ctypes.data, int(pack), sr.ctypes.data,
                          len(sr) // 2, dr.ctypes.data, len(dr) // 2, SMS, -1, 1,
                          ctypes.byref(n))
    assert bad == 0, f"{bad} rows or units outside their buffers / misaligned"


@pytest.mark.parametrize("geo", sorted(GEOS))
def test_emulated_pack_and_unpack_through_a_staging_buffer(emu, geo):
    """The library's own staging side (kvr_staging_desc, as kv_relayout_plan_pack and
    _unpack build it), walked by the emulated kernel: pack equals the oracle's gather
    into [L][C][sum n][H][D], pack then unpack equals the direct relayout."""
    w = _w(3, **GEOS[geo])
    src_bufs = [_aligned(w.src_shape(), np.uint16) for _ in range(w.src_tp)]
    for a, b in zip(src_bufs, w.src_pools_numpy()):
        a[...] = b
    total = int(w.seq_lens.sum())
    stage = _aligned((L_, C_, total, w.kv_heads, w.head_dim), np.uint16)
    stage[...] = 0
    _emu_staging(emu, w, stage, True, src_bufs)
    want = np.zeros_like(stage)
    oracle.relayout_general(_std(w, src_bufs, "src"),
                            [[[want[l, c].reshape(total, 1, w.kv_heads, w.head_dim)
                               for c in range(C_)] for l in range(L_)]],
                            **_tables(_staging_tables(w.geometry(), "dst")))
    np.testing.assert_array_equal(stage, want)
    got_bufs, _ = dst_family(w, "standard")
    _emu_staging(emu, w, stage, False, got_bufs)
    ref = w.dst_pools_numpy()
    oracle.relayout(src_bufs, ref, **w.geometry())
    for a, b in zip(ref, got_bufs):
        np.testing.assert_array_equal(a, b)


# -- validation -----------------------------------------------------------------------

def _fake_layout(base, tp, L, C, view_bytes, bs, ts, hs):
    return dict(bases=[base + i * view_bytes for i in range(tp * L * C)], block_stride=bs,
                token_stride=ts, head_stride=hs)


def test_layout_errors_are_statuses(emu):
    w = _w(4)
    s, d = fake_pools(w)
    L, C, N, B, Hl, D = w.dst_shape()
    row = D * 2
    view = N * B * Hl * row
    good = _fake_layout(1 << 44, w.dst_tp, L, C, view, B * Hl * row, Hl * row, row)
    g = w.geometry()

    def st(dst_layout, src_pools=s):
        return status_of(lambda: kr.desc_bytes(src_pools, None, dst_layout=dst_layout, **g))
    assert st(good) == "KVR_OK"
    assert kr.desc_bytes(s, None, dst_layout=good, **g) == kr.desc_bytes(s, d, **g)
    hnd = _fake_layout(1 << 44, w.dst_tp, L, C, view, B * Hl * row, row, B * row)
    assert st(hnd) == "KVR_OK"
    bad = dict(good, bases=[good["bases"][0] + 8] + good["bases"][1:])
    assert st(bad) == "KVR_ERR_ALIGNMENT"
    assert st(dict(good, token_stride=Hl * row + 8)) == "KVR_ERR_ALIGNMENT"
    assert st(dict(good, block_stride=-16)) == "KVR_ERR_INVALID_ARG"
    assert st(dict(good, bases=[0] + good["bases"][1:])) == "KVR_ERR_INVALID_ARG"
    # rows of one view landing on each other
    assert st(dict(good, head_stride=16)) == "KVR_ERR_POOL_OVERLAP"
    assert st(dict(good, block_stride=Hl * row)) == "KVR_ERR_POOL_OVERLAP"
    # two decode views on top of each other, and a decode view on a prefill pool
    overl = dict(good, bases=[good["bases"][0]] * len(good["bases"]))
    assert st(overl) == "KVR_ERR_POOL_OVERLAP"
    onsrc = dict(good, bases=[s[0]] + good["bases"][1:])
    assert st(onsrc) == "KVR_ERR_POOL_OVERLAP"
    # prefill views may overlap (read only), and the standard pools need not be given
    src_same = _fake_layout(1 << 43, w.src_tp, L, C, 0, *[x * 1 for x in
                                                          (16 * 2 * row, 2 * row, row)])
    assert status_of(lambda: kr.desc_bytes(None, None, src_layout=src_same, dst_layout=good,
                                           **g)) == "KVR_OK"
    # standard pools missing and no layout
    assert status_of(lambda: kr.desc_bytes(None, d, **g)) == "KVR_ERR_INVALID_ARG"


def test_interleaved_views_are_accepted_exactly(emu):
    """K and V interleaved per block ([N][C][B][H][D]) share no byte and pass; the same
    views shifted onto each other by one row are refused."""
    w = _w(5)
    s, _ = fake_pools(w)
    L, C, N, B, Hl, D = w.dst_shape()
    row = D * 2
    blk = B * Hl * row
    base = 1 << 44
    bases = []
    for sh in range(w.dst_tp):
        for l in range(L):
            for c in range(C):
                bases.append(base + (sh * L + l) * N * C * blk + c * blk)
    lay = dict(bases=bases, block_stride=C * blk, token_stride=Hl * row, head_stride=row)
    g = w.geometry()
    assert status_of(lambda: kr.desc_bytes(s, None, dst_layout=lay, **g)) == "KVR_OK"
    shifted = dict(lay, bases=[b - (row if i % 2 else 0) for i, b in enumerate(bases)])
    assert status_of(lambda: kr.desc_bytes(s, None, dst_layout=shifted, **g)) == \
        "KVR_ERR_POOL_OVERLAP"
    # V moved by whole block strides stays in K's gaps (still disjoint) ...
    gaps = dict(lay, bases=[b + 3 * C * blk if i % 2 else b for i, b in enumerate(bases)])
    assert status_of(lambda: kr.desc_bytes(s, None, dst_layout=gaps, **g)) == "KVR_OK"
    # ... but V's first block on K's last block is refused
    last_block = dict(lay, bases=[b + (N - 1) * C * blk - blk if i % 2 else b
                                  for i, b in enumerate(bases)])
    assert status_of(lambda: kr.desc_bytes(s, None, dst_layout=last_block, **g)) == \
        "KVR_ERR_POOL_OVERLAP"


def test_binding_refuses_tensors_smaller_than_the_geometry(emu):
    """The C library sees addresses only; the binding checks that the pools, views
    and staging buffers it is given hold everything the geometry addresses."""
    w = _w(6)
    g = w.geometry()
    src = [_aligned(w.src_shape(), np.uint16) for _ in range(w.src_tp)]
    dst = [_aligned(w.dst_shape(), np.uint16) for _ in range(w.dst_tp)]
    assert kr.desc_bytes(src, dst, **g)[0] > 0
    short = _aligned((int(np.prod(w.dst_shape())) - 1,), np.uint16)
    with pytest.raises(ValueError, match="dst pool 1"):
        kr.desc_bytes(src, [dst[0], short], **g)
    with pytest.raises(ValueError, match="src pool 0 holds"):
        kr.desc_bytes([src[0].reshape(-1)[:-8]] + src[1:], dst, **g)
    with pytest.raises(ValueError, match="src pool 0 is not contiguous"):
        kr.desc_bytes([src[0][:, :, ::2]] + src[1:], dst, **g)
    # views: one block too few, and the wrong element size
    L, C, N, B, Hl, D = w.dst_shape()
    views = [[[b[l, c] for c in range(C)] for l in range(L)] for b in dst]
    assert kr.desc_bytes(src, None, dst_layout=kr.layout_of_views(views), **g)[0] > 0
    fewer = [[[b[l, c][:-1] for c in range(C)] for l in range(L)] for b in dst]
    with pytest.raises(ValueError, match="dst views"):
        kr.desc_bytes(src, None, dst_layout=kr.layout_of_views(fewer), **g)
    wide = [_aligned((L, C, N, B, Hl, D), np.uint32) for _ in range(w.dst_tp)]
    wide_views = [[[b[l, c] for c in range(C)] for l in range(L)] for b in wide]
    with pytest.raises(ValueError, match="4-byte elements"):
        kr.desc_bytes(src, None, dst_layout=kr.layout_of_views(wide_views), **g)
    # staging buffers: the batch's token count, all heads
    total = int(w.seq_lens.sum())
    stage = _aligned((L_, C_, total - 1, w.kv_heads, w.head_dim), np.uint16)
    with pytest.raises(ValueError, match="staging buffer"):
        kr.pack_plan(src, stage, **g)
    with pytest.raises(ValueError, match="staging buffer"):
        kr.pack_plan(src, stage[0], **g)


def test_binding_checks_replicated_pool_extents(emu):
    """With more TP shards than KV heads a shard pool holds one head row per token:
    [L][C][N][B][1][D]; the binding accepts exactly that extent and refuses less."""
    w = _w(7, kv_heads=2, src_tp=4, dst_tp=8, src_block=5, dst_block=16)
    g = w.geometry()
    assert w.src_shape()[4] == 1 and w.dst_shape()[4] == 1
    src = [_aligned(w.src_shape(), np.uint16) for _ in range(w.src_tp)]
    dst = [_aligned(w.dst_shape(), np.uint16) for _ in range(w.dst_tp)]
    r, wr = kr.desc_bytes(src, dst, **g)
    assert wr == 4 * r                                 # every head written to 8 / 2 shards
    short = _aligned((int(np.prod(w.dst_shape())) - 8,), np.uint16)
    with pytest.raises(ValueError, match="dst pool 3"):
        kr.desc_bytes(src, dst[:3] + [short] + dst[4:], **g)

