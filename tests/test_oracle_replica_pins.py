"""Pins of the oracle's head replication (a side with more TP shards than KV heads).

Reading taken (the pages size TP only as a divisor of the head count): with
T > H, T a multiple of H, each KV head is held whole by T/H consecutive
shards, as serving engines replicate KV heads (or an MLA latent) when the TP
degree exceeds them. The hand-off reads a head from the first prefill shard
of its group and writes it to every decode shard of its group.

Checked by meaning (``kvcheck`` reads a request's rows through its blocks,
never through the oracle's shard arithmetic), against the pd.py-style
restatement, and against the unreplicated relayout.
"""
import dataclasses
import itertools

import numpy as np
import pytest

import oracle
from oracle import pd_pages
import workloads as wl
from kvcheck import check_dst, tagged_src

POISON = 0xEEEEEEEE


def _w(name, seed, H, tp, blocks=(16, 32), L=2, C=2, D=3, es=4, lens=(100, 37, 0, 1, 64)):
    return wl.custom(name, seed, num_layers=L, num_components=C, kv_heads=H, head_dim=D,
                     elem_bytes=es, src_tp=tp[0], dst_tp=tp[1], src_block=blocks[0],
                     dst_block=blocks[1], seq_lens=list(lens))


def _poison_later_copies(w, src):
    """Every prefill shard but the first of each head's group holds only poison."""
    if w.src_tp > w.kv_heads:
        group = w.src_tp // w.kv_heads
        for s, pool in enumerate(src):
            if s % group:
                pool[...] = w._sentinel_value(0xEE)
    return src


REPLICATED_TP = [(tp_s, tp_d) for tp_s, tp_d in itertools.product([1, 2, 4, 8], [1, 2, 4, 8])
                 if tp_s > 2 or tp_d > 2]


@pytest.mark.parametrize("tp", REPLICATED_TP)
@pytest.mark.parametrize("H", [1, 2])
def test_tagged_heads_reach_every_decode_copy_from_the_first_prefill_copy(oracle_lib, H, tp):
    """Tags (unique per element) written to every prefill copy, then all copies but the
    first of each group poisoned: every decode copy of every head holds that head's
    tags in the request's slots, and nothing else changed."""
    if tp[0] < H and H % tp[0] or tp[1] < H and H % tp[1]:
        pytest.skip("TP neither divides nor is a multiple of H")
    for blocks in ((16, 32), (3, 5), (64, 1)):
        w = _w(f"rep{H}_{tp}_{blocks}", 500 + H * 10 + tp[0] + tp[1], H, tp, blocks)
        src, expected = tagged_src(w, poison=POISON)
        _poison_later_copies(w, src)
        dst = w.dst_pools_numpy()
        oracle.relayout(src, dst, lib=oracle_lib, **w.geometry())
        check_dst(w, dst, expected, w._sentinel_value(0xFF))


@pytest.mark.parametrize("H,tp", [(1, (1, 8)), (1, (8, 1)), (1, (4, 4)), (2, (1, 8)),
                                  (2, (8, 2)), (4, (8, 16)), (8, (4, 16)), (8, (16, 2))])
def test_pd_py_restatement_agrees_with_replication(oracle_lib, H, tp):
    """Random bits, copies drawn independently: the C loop nest equals pd.py's gather
    (first copy of each head) and admit (every copy of each head)."""
    w = _w(f"pdrep{H}_{tp}", 600 + H + tp[0] * 3 + tp[1], H, tp, (16, 64), L=2, C=2, D=8,
           es=2, lens=(150, 64, 1))
    src = w.src_pools_numpy()
    a, b = w.dst_pools_numpy(), w.dst_pools_numpy()
    oracle.relayout(src, a, lib=oracle_lib, **w.geometry())
    pd_pages.relayout(src, b, **w.geometry())
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("H,tp_d", [(1, 4), (2, 4), (8, 16), (4, 8)])
def test_decode_copies_equal_the_unreplicated_relayout(oracle_lib, H, tp_d):
    """Decode TP = k*H: every copy k of head h equals shard h of the same relayout with
    decode TP = H (one head per shard, no copies)."""
    w = _w(f"cp{H}_{tp_d}", 700 + H + tp_d, H, (1, tp_d), (16, 32), D=8, es=2)
    base = dataclasses.replace(w, name=w.name + "_base", dst_tp=H)
    src = w.src_pools_numpy()
    got, ref = w.dst_pools_numpy(), base.dst_pools_numpy()
    oracle.relayout(src, got, lib=oracle_lib, **w.geometry())
    oracle.relayout(src, ref, lib=oracle_lib, **base.geometry())
    group = tp_d // H
    for s, pool in enumerate(got):
        np.testing.assert_array_equal(pool, ref[s // group], err_msg=f"decode shard {s}")


@pytest.mark.parametrize("H,tp_s", [(1, 4), (2, 8), (8, 16)])
def test_prefill_copies_reduce_to_the_first_copy(oracle_lib, H, tp_s):
    """Prefill TP = k*H, later copies poisoned: the result equals the relayout from
    prefill TP = H over the first copies alone."""
    w = _w(f"pc{H}_{tp_s}", 800 + H + tp_s, H, (tp_s, 1), (16, 32), D=8, es=2)
    first_only = dataclasses.replace(w, name=w.name + "_first", src_tp=H)
    src = _poison_later_copies(w, w.src_pools_numpy())
    group = tp_s // H
    got, ref = w.dst_pools_numpy(), first_only.dst_pools_numpy()
    oracle.relayout(src, got, lib=oracle_lib, **w.geometry())
    oracle.relayout(src[::group], ref, lib=oracle_lib, **first_only.geometry())
    for x, y in zip(got, ref):
        np.testing.assert_array_equal(x, y)


def test_replication_in_the_converting_and_layout_nests(oracle_lib):
    """The converting and the layout-generic loop nests replicate the same way: with
    standard views they equal the converting oracle, and a bit-copy general relayout
    equals the plain one (decode copies and poisoned prefill copies included)."""
    w = _w("convrep", 901, 2, (4, 8), (16, 32), D=16, es=2, lens=(70, 33))
    rng = np.random.default_rng(5)
    src = _poison_later_copies(w, [rng.integers(0, 1 << 16, w.src_shape(), dtype=np.uint16)
                                   for _ in range(w.src_tp)])
    geo = w.geometry()
    tables = {k: geo[k] for k in ("num_layers", "num_components", "kv_heads", "head_dim",
                                  "src_tp", "dst_tp", "src_block", "dst_block", "seq_lens",
                                  "src_off", "src_bt", "dst_off", "dst_bt")}
    Hs = wl.heads_per_shard(w.kv_heads, w.src_tp)
    Hd = wl.heads_per_shard(w.kv_heads, w.dst_tp)
    sv = oracle.standard_views(src, w.num_layers, 2, w.src_num_blocks, w.src_block, Hs,
                               w.head_dim)
    plain = w.dst_pools_numpy()
    oracle.relayout(src, plain, lib=oracle_lib, **geo)
    gen = w.dst_pools_numpy()
    dv = oracle.standard_views(gen, w.num_layers, 2, w.dst_num_blocks, w.dst_block, Hd,
                               w.head_dim)
    oracle.relayout_general(sv, dv, lib=oracle_lib, **tables)
    for x, y in zip(plain, gen):
        np.testing.assert_array_equal(x, y)
    scales = rng.uniform(0.01, 2.0, w.num_layers * 2 * w.kv_heads).astype(np.float32)
    q_std = [np.full(w.dst_shape(), 0xFF, np.uint8) for _ in range(w.dst_tp)]
    g2 = dict(geo)
    g2.pop("elem_bytes")
    oracle.relayout_convert(src, q_std, lib=oracle_lib, src_dtype=oracle.BF16,
                            dst_dtype=oracle.E4M3, per_head=1, scales=scales, **g2)
    q_gen = [np.full(w.dst_shape(), 0xFF, np.uint8) for _ in range(w.dst_tp)]
    qv = oracle.standard_views(q_gen, w.num_layers, 2, w.dst_num_blocks, w.dst_block, Hd,
                               w.head_dim)
    oracle.relayout_general(sv, qv, lib=oracle_lib, src_dtype=oracle.BF16,
                            dst_dtype=oracle.E4M3, per_head=1, scales=scales, **tables)
    for x, y in zip(q_std, q_gen):
        np.testing.assert_array_equal(x, y)
    # and the copies of the converting nest agree among themselves
    for s in range(0, w.dst_tp, 2):
        np.testing.assert_array_equal(q_std[s], q_std[s + 1])


def test_tp_that_neither_divides_nor_multiplies_is_refused(oracle_lib):
    w = _w("bad", 950, 4, (1, 1))
    for tp in ((3, 1), (1, 6), (8, 3)):
        bad = dataclasses.replace(w, src_tp=tp[0], dst_tp=tp[1])
        with pytest.raises(Exception):
            oracle.relayout([np.zeros(8, np.uint32)] * tp[0], [np.zeros(8, np.uint32)] * tp[1],
                            lib=oracle_lib, **bad.geometry())
