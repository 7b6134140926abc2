"""Test helpers that read and write paged pools by what a block table MEANS.

A request's KV, for one layer and component, is its physical blocks laid end
to end in table order, cut at the prompt length; the TP shards of one side
hold consecutive head ranges, laid side by side along the head axis (with more
shards than heads, each group of T/H consecutive shards holds one head: any
one of them, ``replica``, gives that head's rows). These
helpers use only that meaning (numpy reshapes and fancy indexing over whole
blocks), never the per-token slot arithmetic, so they can judge both the
oracle and the CUDA path without repeating either's index expressions.
"""
from __future__ import annotations

import numpy as np


def copies(pools, kv_heads):
    """Shards that hold one head (1 unless a side has more shards than heads)."""
    if kv_heads is None or len(pools) <= kv_heads:
        return 1
    return len(pools) // kv_heads


def request_rows(pools, shape, layer, comp, ids, n, kv_heads=None, replica=0):
    """Tokens [0, n) of one request as [n, H, D] (shards side by side; of each group
    of shards holding the same head, the ``replica``-th)."""
    L, C, N, B, Hl, D = shape
    parts = []
    for pool in pools[replica::copies(pools, kv_heads)]:
        v = pool.reshape(shape)
        parts.append(v[layer, comp][np.asarray(ids, dtype=np.int64)].reshape(-1, Hl, D)[:n])
    return np.concatenate(parts, axis=1)


def write_request_rows(pools, shape, layer, comp, ids, rows, kv_heads=None):
    """Inverse of :func:`request_rows`: put [n, H, D] rows into the request's blocks
    (every shard of a group holding the same head gets it)."""
    L, C, N, B, Hl, D = shape
    ids = np.asarray(ids, dtype=np.int64)
    n = rows.shape[0]
    g = copies(pools, kv_heads)
    for s, pool in enumerate(pools):
        v = pool.reshape(shape)
        buf = v[layer, comp][ids].reshape(len(ids) * B, Hl, D)
        first = (s // g) * Hl
        buf[:n] = rows[:, first:first + Hl]
        v[layer, comp][ids] = buf.reshape(len(ids), B, Hl, D)


def covered_mask(shape, off, bt, lens):
    """Boolean [N, B]: the (block, offset) slots that hold some request's prompt token."""
    L, C, N, B, Hl, D = shape
    m = np.zeros((N, B), dtype=bool)
    for r, n in enumerate(np.asarray(lens).tolist()):
        if n == 0:
            continue
        ids = np.asarray(bt[off[r]:off[r + 1]], dtype=np.int64)
        nb = -(-n // B)
        ids = ids[:nb]
        tmp = m[ids].reshape(-1)
        tmp[:n] = True
        m[ids] = tmp.reshape(nb, B)
    return m


def full_mask(shape, slot_mask):
    L, C, N, B, Hl, D = shape
    return np.broadcast_to(slot_mask[None, None, :, :, None, None], shape)


def src_ids(w, r):
    return w.src_bt[w.src_off[r]:w.src_off[r + 1]]


def dst_ids(w, r):
    return w.dst_bt[w.dst_off[r]:w.dst_off[r + 1]]


def tagged_src(w, poison):
    """Prefill pools whose prompt elements carry unique tags 1, 2, 3, ...

    Every other element holds ``poison``. Returns (pools, expected) with
    expected[r] of shape [L, C, n_r, H, D].
    """
    dt = w.int_dtype()
    pools = [np.full(w.src_shape(), poison, dtype=dt) for _ in range(w.src_tp)]
    expected, nxt = [], 1
    for r, n in enumerate(w.seq_lens.tolist()):
        cnt = w.num_layers * w.num_components * n * w.kv_heads * w.head_dim
        tags = (np.arange(cnt, dtype=np.int64) + nxt)
        nxt += cnt
        if nxt >= min(int(np.iinfo(dt).max), poison):
            raise ValueError("too many elements to tag in this element width")
        tags = tags.astype(dt).reshape(w.num_layers, w.num_components, n, w.kv_heads,
                                       w.head_dim)
        expected.append(tags)
        if n == 0:
            continue
        for l in range(w.num_layers):
            for c in range(w.num_components):
                write_request_rows(pools, w.src_shape(), l, c, src_ids(w, r), tags[l, c],
                                   w.kv_heads)
    return pools, expected


def expected_from_src(w, src_pools, layers=None):
    """What each request's decode rows must hold: its prefill rows, by meaning."""
    layers = range(w.num_layers) if layers is None else layers
    out = []
    for r, n in enumerate(w.seq_lens.tolist()):
        rows = np.zeros((w.num_layers, w.num_components, n, w.kv_heads, w.head_dim),
                        dtype=w.int_dtype())
        if n:
            for l in layers:
                for c in range(w.num_components):
                    rows[l, c] = request_rows(src_pools, w.src_shape(), l, c, src_ids(w, r), n,
                                              w.kv_heads)
        out.append(rows)
    return out


def check_dst(w, dst_pools, expected, sentinel, layers=None):
    """Assert every prompt row sits where the decode table says and nothing else changed."""
    layers = list(range(w.num_layers)) if layers is None else list(layers)
    for r, n in enumerate(w.seq_lens.tolist()):
        if n == 0:
            continue
        for l in layers:
            for c in range(w.num_components):
                for k in range(copies(dst_pools, w.kv_heads)):
                    got = request_rows(dst_pools, w.dst_shape(), l, c, dst_ids(w, r), n,
                                       w.kv_heads, replica=k)
                    np.testing.assert_array_equal(
                        got, expected[r][l, c], err_msg=f"request {r} layer {l} comp {c} "
                                                        f"copy {k}")
    slot = covered_mask(w.dst_shape(), w.dst_off, w.dst_bt, w.seq_lens)
    cover = full_mask(w.dst_shape(), slot)
    for pool in dst_pools:
        v = pool.reshape(w.dst_shape())
        for l in range(w.num_layers):
            if l in layers:
                untouched = v[l][~cover[l]]
            else:
                untouched = v[l].reshape(-1)
            assert np.all(untouched == sentinel), f"layer {l}: bytes outside the prompt changed"
