"""Pins of the CPU oracle to what the pages and the mathematics fix.

None of these checks repeats the oracle's index expressions: decode-side
results are read back by what a block table means (``kvcheck``), values are
compared against figures the pages print, against a second restatement staged
like pd.py, against the relayout's own inverse, and against a plain copy.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import pd_pages
import workloads as wl
from kvcheck import check_dst, covered_mask, expected_from_src, full_mask, tagged_src

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")


def _run(w, src, dst, lib=None, **kw):
    oracle.relayout(src, dst, lib=lib, **w.geometry(), **kw)


def _sentinel(w, byte=0xFF):
    return w._sentinel_value(byte)


# -- byte counts the pages print ------------------------------------------------

def _figs():
    with open(GOLDEN) as f:
        return json.load(f)


def _bpt(shape, lib):
    return oracle.bytes_per_token(shape["L"], shape["C"], shape["H"], shape["D"], shape["es"],
                                  lib=lib)


def test_llama70b_4k_prompt_is_1_34_gb_and_27_ms(oracle_lib):
    g = _figs()["llama3_70b_4k"]
    assert _bpt(g["shape"], oracle_lib) == 320 * 1024 == g["per_token_bytes"]
    s = g["shape"]
    total = oracle.transfer_bytes(s["L"], s["C"], s["H"], s["D"], s["es"], g["prompt_lens"],
                                  lib=oracle_lib)
    assert total == 1_342_177_280
    assert f"{total / 1e9:.2f}" == g["printed_gb_2dp"]
    assert round(total / g["link_bytes_per_s"] * 1e3) == g["printed_link_ms"]


def test_deepseek_mla_4k_prompt_is_0_29_gb_and_6_ms(oracle_lib):
    g = _figs()["deepseek_v3_mla_4k"]
    assert _bpt(g["shape"], oracle_lib) == g["per_token_bytes"] == 70272
    s = g["shape"]
    total = oracle.transfer_bytes(s["L"], s["C"], s["H"], s["D"], s["es"], g["prompt_lens"],
                                  lib=oracle_lib)
    assert total == 287_834_112
    assert f"{total / 1e9:.2f}" == g["printed_gb_2dp"]
    assert round(total / g["link_bytes_per_s"] * 1e3) == g["printed_link_ms"]


def test_qwen3_32b_is_256_kb_per_token(oracle_lib):
    g = _figs()["qwen3_32b_per_token"]
    assert _bpt(g["shape"], oracle_lib) == g["per_token_printed_kb"] * 1024


def test_pd_demo_moves_7840_kb_for_70_tokens(oracle_lib):
    g = _figs()["pd_demo_70_tokens"]
    s = g["shape"]
    # the split of the 70 tokens over the 4 prompts does not matter: the count is linear
    for lens in ([70], [17, 18, 17, 18], [1, 1, 1, 67]):
        assert sum(lens) == g["prompt_tokens_total"]
        total = oracle.transfer_bytes(s["L"], s["C"], s["H"], s["D"], s["es"], lens,
                                      lib=oracle_lib)
        assert f"{total / 1024:.0f}" == str(g["printed_kb"])


def test_exercise5_needs_13_1_gb_per_s(oracle_lib):
    g = _figs()["cs349d_ex5"]
    s = g["shape"]
    per_s = oracle.transfer_bytes(s["L"], s["C"], s["H"], s["D"], s["es"],
                                  [g["prompt_len"]] * g["requests_per_s"], lib=oracle_lib)
    assert f"{per_s / 1e9:.1f}" == g["printed_gb_per_s_1dp"]


def test_relayout_moves_exactly_the_counted_bytes(oracle_lib):
    """Two runs over pools pre-filled with different sentinels: an element the
    relayout wrote is equal in both, an untouched one differs. Their count times
    the element size must be the page's KV/token x prompt length."""
    for w in (wl.tiny(),
              wl.custom("c", 11, num_layers=3, num_components=2, kv_heads=6, head_dim=8,
                        elem_bytes=2, src_tp=3, dst_tp=2, src_block=5, dst_block=7,
                        seq_lens=[0, 1, 33, 70, 7])):
        src = w.src_pools_numpy()
        a = w.dst_pools_numpy(0xFF)
        b = w.dst_pools_numpy(0xAA)
        _run(w, src, a, lib=oracle_lib)
        _run(w, src, b, lib=oracle_lib)
        written = sum(int(np.count_nonzero(x == y)) for x, y in zip(a, b))
        assert written * w.elem_bytes == oracle.transfer_bytes(
            w.num_layers, w.num_components, w.kv_heads, w.head_dim, w.elem_bytes, w.seq_lens,
            lib=oracle_lib)


# -- placement: brute force with tags ------------------------------------------------

def test_tiny_tagged_every_tag_lands_once_in_its_decode_slot(oracle_lib):
    w = wl.tiny()
    src, expected = tagged_src(w, poison=0xEEEE)
    dst = w.dst_pools_numpy()
    _run(w, src, dst, lib=oracle_lib)
    check_dst(w, dst, expected, _sentinel(w))
    # each tag appears exactly once in the whole decode pool
    vals = np.concatenate([p.reshape(-1) for p in dst])
    vals = vals[vals != 0xFFFF]
    assert len(vals) == 2 * 2 * 100 * 2 * 64
    assert len(np.unique(vals)) == len(vals)


@pytest.mark.parametrize("tp", list(itertools.product([1, 2], [1, 2])))
def test_enumerate_block_sizes_and_tp(oracle_lib, tp):
    """All (Bp, Bd) in {1..64}^2 x (Tp, Td) in {1,2}^2 with H = 2, tagged."""
    sizes = [1, 2, 4, 8, 16, 32, 64]
    for bp, bd in itertools.product(sizes, sizes):
        w = wl.custom(f"e{bp}_{bd}", 100 + bp * 7 + bd, num_layers=2, num_components=2,
                      kv_heads=2, head_dim=3, elem_bytes=4, src_tp=tp[0], dst_tp=tp[1],
                      src_block=bp, dst_block=bd, seq_lens=[100, 37, 0, 1, 64])
        src, expected = tagged_src(w, poison=0xEEEEEEEE)
        dst = w.dst_pools_numpy()
        _run(w, src, dst, lib=oracle_lib)
        check_dst(w, dst, expected, _sentinel(w))


def test_random_bits_land_where_tags_do(oracle_lib):
    """Value independence: random bit patterns (NaN payloads included) move bit-exactly."""
    w = wl.tiny()
    src = w.src_pools_numpy()
    dst = w.dst_pools_numpy()
    _run(w, src, dst, lib=oracle_lib)
    check_dst(w, dst, expected_from_src(w, src), _sentinel(w))


# -- inverse, plain copy, modes ------------------------------------------------------

def _swap_roles(w, name):
    """The decode side as a source and a fresh prefill-shaped pool as destination."""
    import dataclasses
    return dataclasses.replace(w, name=name, src_tp=w.dst_tp, dst_tp=w.src_tp,
                               src_block=w.dst_block, dst_block=w.src_block,
                               src_num_blocks=w.dst_num_blocks, dst_num_blocks=w.src_num_blocks,
                               src_off=w.dst_off, src_bt=w.dst_bt, dst_off=w.src_off,
                               dst_bt=w.src_bt)


@pytest.mark.parametrize("case", ["tp4_to_tp8", "tp4_to_tp2_ragged", "tp3_to_tp2_odd_blocks"])
def test_relayout_then_inverse_is_identity(oracle_lib, case):
    if case == "tp4_to_tp8":
        w = wl.custom(case, 21, num_layers=2, num_components=2, kv_heads=8, head_dim=16,
                      elem_bytes=2, src_tp=4, dst_tp=8, src_block=16, dst_block=32,
                      seq_lens=[4096])
    elif case == "tp4_to_tp2_ragged":
        w = wl.custom(case, 22, num_layers=2, num_components=2, kv_heads=8, head_dim=16,
                      elem_bytes=2, src_tp=4, dst_tp=2, src_block=16, dst_block=64,
                      seq_lens=[1000 - 5, 1000 - 63, 1000 - 1, 1000 - 32])
    else:
        w = wl.custom(case, 23, num_layers=3, num_components=2, kv_heads=6, head_dim=4,
                      elem_bytes=2, src_tp=3, dst_tp=2, src_block=3, dst_block=5,
                      seq_lens=[17, 0, 1, 29])
    src = w.src_pools_numpy()
    mid = w.dst_pools_numpy(0xFF)
    _run(w, src, mid, lib=oracle_lib)
    back_w = _swap_roles(w, case + "_inv")
    back = back_w.dst_pools_numpy(0xAA)
    oracle.relayout(mid, back, lib=oracle_lib, **back_w.geometry())
    slot = covered_mask(w.src_shape(), w.src_off, w.src_bt, w.seq_lens)
    cover = full_mask(w.src_shape(), slot)
    for s, (orig, got) in enumerate(zip(src, back)):
        np.testing.assert_array_equal(got[cover], orig[cover], err_msg=f"shard {s}")
        assert np.all(got[~cover] == 0xAAAA)


def test_equal_blocks_equal_tp_identity_tables_is_a_plain_copy(oracle_lib):
    n, B, N = 1000, 16, 80
    ids = np.arange(N, dtype=np.int32)
    lens = np.array([n], np.int32)
    off = np.array([0, N], np.int64)
    import dataclasses
    base = wl.custom("copy", 31, num_layers=3, num_components=2, kv_heads=4, head_dim=8,
                     elem_bytes=2, src_tp=2, dst_tp=2, src_block=B, dst_block=B, seq_lens=[n],
                     src_num_blocks=N, dst_num_blocks=N)
    w = dataclasses.replace(base, seq_lens=lens, src_off=off, src_bt=ids, dst_off=off, dst_bt=ids)
    src = w.src_pools_numpy()
    dst = w.dst_pools_numpy()
    _run(w, src, dst, lib=oracle_lib)
    for s, d in zip(src, dst):
        L, C, _, _, Hl, D = w.src_shape()
        sflat = s.reshape(L, C, N * B * Hl * D)
        dflat = d.reshape(L, C, N * B * Hl * D)
        cut = n * Hl * D
        np.testing.assert_array_equal(dflat[:, :, :cut], sflat[:, :, :cut])
        assert np.all(dflat[:, :, cut:] == 0xFFFF)


def test_layer_by_layer_equals_whole_prompt(oracle_lib):
    w = wl.custom("modes", 41, num_layers=4, num_components=2, kv_heads=4, head_dim=8,
                  elem_bytes=2, src_tp=2, dst_tp=4, src_block=16, dst_block=32,
                  seq_lens=[300, 5, 77])
    src = w.src_pools_numpy()
    whole = w.dst_pools_numpy()
    _run(w, src, whole, lib=oracle_lib)
    per = w.dst_pools_numpy()
    for l in range(w.num_layers):
        _run(w, src, per, lib=oracle_lib, layer_begin=l, layer_end=l + 1)
    for a, b in zip(whole, per):
        np.testing.assert_array_equal(a, b)


def test_single_layer_slice_equals_layer_of_whole(oracle_lib):
    """A layer's slice of the pools, run as a one-layer problem, gives that layer's result
    (used to stream the large configurations one layer at a time)."""
    import dataclasses
    w = wl.custom("slice", 42, num_layers=3, num_components=2, kv_heads=8, head_dim=8,
                  elem_bytes=2, src_tp=4, dst_tp=2, src_block=16, dst_block=64,
                  seq_lens=[200, 65])
    src = w.src_pools_numpy()
    whole = w.dst_pools_numpy()
    _run(w, src, whole, lib=oracle_lib)
    w1 = dataclasses.replace(w, num_layers=1)
    for l in range(w.num_layers):
        s1 = [np.ascontiguousarray(p[l:l + 1]) for p in src]
        d1 = w1.dst_pools_numpy()
        _run(w1, s1, d1, lib=oracle_lib)
        for a, b in zip(whole, d1):
            np.testing.assert_array_equal(a[l:l + 1], b)


def test_empty_batch_and_zero_length_prompts_touch_nothing(oracle_lib):
    w = wl.custom("empty", 51, num_layers=2, num_components=2, kv_heads=2, head_dim=8,
                  elem_bytes=2, src_tp=1, dst_tp=2, src_block=4, dst_block=8,
                  seq_lens=[0, 0, 0])
    src = w.src_pools_numpy()
    dst = w.dst_pools_numpy()
    _run(w, src, dst, lib=oracle_lib)
    assert all(np.all(d == 0xFFFF) for d in dst)


# -- the two restatements agree ----------------------------------------------------

@pytest.mark.parametrize("spec", [
    dict(kv_heads=2, src_tp=1, dst_tp=1, src_block=16, dst_block=32, lens=[100]),
    dict(kv_heads=8, src_tp=4, dst_tp=8, src_block=16, dst_block=32, lens=[333, 1, 64]),
    dict(kv_heads=8, src_tp=4, dst_tp=2, src_block=16, dst_block=64, lens=[250, 0, 129]),
    dict(kv_heads=12, src_tp=3, dst_tp=2, src_block=3, dst_block=5, lens=[40, 17]),
    dict(kv_heads=6, src_tp=2, dst_tp=3, src_block=64, dst_block=16, lens=[300, 64, 65]),
    dict(kv_heads=1, src_tp=1, dst_tp=1, src_block=64, dst_block=16, lens=[129, 1000]),
])
def test_c_loop_nest_agrees_with_pd_py_staging(oracle_lib, spec):
    w = wl.custom("agree", 61, num_layers=2, num_components=2, kv_heads=spec["kv_heads"],
                  head_dim=8, elem_bytes=2, src_tp=spec["src_tp"], dst_tp=spec["dst_tp"],
                  src_block=spec["src_block"], dst_block=spec["dst_block"],
                  seq_lens=spec["lens"], shared_prefix=2)
    src = w.src_pools_numpy()
    a = w.dst_pools_numpy()
    b = w.dst_pools_numpy()
    _run(w, src, a, lib=oracle_lib)
    pd_pages.relayout(src, b, **w.geometry())
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    check_dst(w, a, expected_from_src(w, src), 0xFFFF)


def test_shared_prefix_blocks_are_read_by_every_request(oracle_lib):
    w = wl.custom("prefix", 71, num_layers=2, num_components=2, kv_heads=4, head_dim=8,
                  elem_bytes=2, src_tp=2, dst_tp=1, src_block=16, dst_block=32,
                  seq_lens=[100, 90, 64], shared_prefix=3)
    assert np.array_equal(w.src_bt[w.src_off[1]:w.src_off[1] + 3], w.src_bt[:3])
    src = w.src_pools_numpy()
    dst = w.dst_pools_numpy()
    _run(w, src, dst, lib=oracle_lib)
    check_dst(w, dst, expected_from_src(w, src), 0xFFFF)
