"""Pins of the oracle's layout-generic relayout.

A layout is given per (shard, layer, component) as a strided view
[block][token][head][dim]. The pins never restate the oracle's address
expression: the expected results come from the already-pinned standard-layout
oracles, with numpy doing the layout changes (transposes, separate buffers,
interleaving), and from pd.py's gather (``oracle.pd_pages``) for the staging
buffer.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from oracle import pd_pages
import workloads as wl


def _w(seed, **kw):
    base = dict(num_layers=3, num_components=2, kv_heads=8, head_dim=16, elem_bytes=2,
                src_tp=4, dst_tp=2, src_block=16, dst_block=64, seq_lens=[300, 1, 77, 0])
    base.update(kw)
    return wl.custom("layout", seed, **base)


def _std_views(w, pools, side):
    if side == "src":
        return oracle.standard_views(pools, w.num_layers, w.num_components, w.src_num_blocks,
                                     w.src_block, w.kv_heads // w.src_tp, w.head_dim)
    return oracle.standard_views(pools, w.num_layers, w.num_components, w.dst_num_blocks,
                                 w.dst_block, w.kv_heads // w.dst_tp, w.head_dim)


def _tables(w):
    return dict(num_layers=w.num_layers, num_components=w.num_components, kv_heads=w.kv_heads,
                head_dim=w.head_dim, src_tp=w.src_tp, dst_tp=w.dst_tp, src_block=w.src_block,
                dst_block=w.dst_block, seq_lens=w.seq_lens, src_off=w.src_off, src_bt=w.src_bt,
                dst_off=w.dst_off, dst_bt=w.dst_bt)


def _standard_result(w, src, lib):
    ref = w.dst_pools_numpy()
    oracle.relayout(src, ref, lib=lib, **w.geometry())
    return ref


def test_standard_views_reduce_to_the_standard_oracle(oracle_lib):
    for w in (_w(1), _w(2, kv_heads=6, src_tp=3, dst_tp=2, src_block=3, dst_block=5,
                    elem_bytes=4, seq_lens=[40, 0, 17])):
        src = w.src_pools_numpy()
        ref = _standard_result(w, src, oracle_lib)
        got = w.dst_pools_numpy()
        oracle.relayout_general(_std_views(w, src, "src"), _std_views(w, got, "dst"),
                                lib=oracle_lib, **_tables(w))
        for a, b in zip(ref, got):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("direction", ["quant", "dequant"])
def test_standard_views_reduce_to_the_converting_oracle(oracle_lib, direction):
    rng = np.random.default_rng(3)
    w = _w(4, elem_bytes=2 if direction == "quant" else 1)
    if direction == "quant":
        src = [rng.integers(0, 1 << 16, w.src_shape(), dtype=np.uint16) for _ in range(4)]
        kw = dict(src_dtype=oracle.BF16, dst_dtype=oracle.E4M3)
        dst_dt = np.uint8
    else:
        src = [rng.integers(0, 256, w.src_shape(), dtype=np.uint8) for _ in range(4)]
        kw = dict(src_dtype=oracle.E4M3, dst_dtype=oracle.BF16)
        dst_dt = np.uint16
    scales = rng.uniform(0.01, 3.0, w.num_layers * 2 * 8).astype(np.float32)
    ref = [np.zeros(w.dst_shape(), dst_dt) for _ in range(2)]
    g = w.geometry()
    g.pop("elem_bytes")
    oracle.relayout_convert(src, ref, per_head=1, scales=scales, lib=oracle_lib, **kw, **g)
    got = [np.zeros(w.dst_shape(), dst_dt) for _ in range(2)]
    oracle.relayout_general(_std_views(w, src, "src"), _std_views(w, got, "dst"), per_head=1,
                            scales=scales, lib=oracle_lib, **kw, **_tables(w))
    for a, b in zip(ref, got):
        np.testing.assert_array_equal(a, b)


def _hnd_dst(w):
    """Decode pools stored head-major inside each block: [L][C][N][H/T][B][D]."""
    L, C, N, B, Hl, D = w.dst_shape()
    pools = [np.full((L, C, N, Hl, B, D), 0xFFFF, np.uint16) for _ in range(w.dst_tp)]
    views = [[[p[l, c].transpose(0, 2, 1, 3) for c in range(C)] for l in range(L)]
             for p in pools]
    return pools, views


def test_head_major_blocks_are_a_transpose(oracle_lib):
    w = _w(5)
    src = w.src_pools_numpy()
    ref = _standard_result(w, src, oracle_lib)
    pools, views = _hnd_dst(w)
    oracle.relayout_general(_std_views(w, src, "src"), views, lib=oracle_lib, **_tables(w))
    for a, p in zip(ref, pools):
        np.testing.assert_array_equal(np.ascontiguousarray(p.transpose(0, 1, 2, 4, 3, 5)), a)


def test_head_major_prefill_side_too(oracle_lib):
    w = _w(6)
    src = w.src_pools_numpy()
    ref = _standard_result(w, src, oracle_lib)
    hnd = [np.ascontiguousarray(s.transpose(0, 1, 2, 4, 3, 5)) for s in src]   # [L][C][N][H][B][D]
    L, C = w.num_layers, w.num_components
    sviews = [[[p[l, c].transpose(0, 2, 1, 3) for c in range(C)] for l in range(L)] for p in hnd]
    got = w.dst_pools_numpy()
    oracle.relayout_general(sviews, _std_views(w, got, "dst"), lib=oracle_lib, **_tables(w))
    for a, b in zip(ref, got):
        np.testing.assert_array_equal(a, b)


def test_separate_buffers_per_layer_and_component(oracle_lib):
    """Every (shard, layer, K/V) its own buffer, as engines that keep one K and one V
    tensor per layer do."""
    w = _w(7)
    src = w.src_pools_numpy()
    ref = _standard_result(w, src, oracle_lib)
    L, C, N, B, Hl, D = w.dst_shape()
    bufs = [[[np.full((N, B, Hl, D), 0xFFFF, np.uint16) for _ in range(C)] for _ in range(L)]
            for _ in range(w.dst_tp)]
    oracle.relayout_general(_std_views(w, src, "src"), bufs, lib=oracle_lib, **_tables(w))
    for s in range(w.dst_tp):
        for l in range(L):
            for c in range(C):
                np.testing.assert_array_equal(bufs[s][l][c], ref[s][l, c])


def test_k_and_v_interleaved_per_block(oracle_lib):
    """[L][N][C][B][H][D]: the K and V of a block next to each other."""
    w = _w(8)
    src = w.src_pools_numpy()
    ref = _standard_result(w, src, oracle_lib)
    L, C, N, B, Hl, D = w.dst_shape()
    pools = [np.full((L, N, C, B, Hl, D), 0xFFFF, np.uint16) for _ in range(w.dst_tp)]
    views = [[[p[l, :, c] for c in range(C)] for l in range(L)] for p in pools]
    oracle.relayout_general(_std_views(w, src, "src"), views, lib=oracle_lib, **_tables(w))
    for a, p in zip(ref, pools):
        np.testing.assert_array_equal(np.ascontiguousarray(p.transpose(0, 2, 1, 3, 4, 5)), a)


def _staging(w):
    """A contiguous [L][C][sum n][H][D] buffer seen as one-token blocks (one shard)."""
    total = int(w.seq_lens.sum())
    buf = np.zeros((w.num_layers, w.num_components, total, w.kv_heads, w.head_dim), np.uint16)
    views = [[[buf[l, c].reshape(total, 1, w.kv_heads, w.head_dim)
               for c in range(w.num_components)] for l in range(w.num_layers)]]
    off = np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int64)
    ids = np.arange(total, dtype=np.int32)
    return buf, views, off, ids


def test_staging_buffer_holds_pd_py_gather(oracle_lib):
    """Packing into [L][C][tokens][H][D] gives, request by request, exactly what pd.py's
    prefill() gathers per layer: [seq, kv_heads, head_dim] of K and of V."""
    w = _w(9)
    src = w.src_pools_numpy()
    buf, views, off, ids = _staging(w)
    t = _tables(w)
    t.update(dst_tp=1, dst_block=1, dst_off=off, dst_bt=ids)
    oracle.relayout_general(_std_views(w, src, "src"), views, lib=oracle_lib, **t)
    for r, n in enumerate(w.seq_lens.tolist()):
        if n == 0:
            continue
        blocks = w.src_bt[w.src_off[r]:w.src_off[r + 1]][: -(-n // w.src_block)]
        for l in range(w.num_layers):
            for c in range(w.num_components):
                want = pd_pages.gather_prefill(src, l, c, blocks, n, num_layers=w.num_layers,
                                               num_components=w.num_components,
                                               kv_heads=w.kv_heads, head_dim=w.head_dim,
                                               src_tp=w.src_tp, src_block=w.src_block,
                                               src_num_blocks=w.src_num_blocks)
                np.testing.assert_array_equal(buf[l, c, off[r]:off[r] + n], want)


def test_pack_then_unpack_equals_the_direct_relayout(oracle_lib):
    w = _w(10)
    src = w.src_pools_numpy()
    ref = _standard_result(w, src, oracle_lib)
    buf, views, off, ids = _staging(w)
    t = _tables(w)
    t.update(dst_tp=1, dst_block=1, dst_off=off, dst_bt=ids)
    oracle.relayout_general(_std_views(w, src, "src"), views, lib=oracle_lib, **t)
    got = w.dst_pools_numpy()
    t = _tables(w)
    t.update(src_tp=1, src_block=1, src_off=off, src_bt=ids)
    oracle.relayout_general(views, _std_views(w, got, "dst"), lib=oracle_lib, **t)
    for a, b in zip(ref, got):
        np.testing.assert_array_equal(a, b)
