"""Second CPU definition of the KV hand-off, staged the way pd.py stages it.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``). Small inputs only.

Page "PD 分离与 KV 传输" (ai-infra-handbooks, serving/distributed/pd-disagg),
section "实现": the prefill instance's ``prefill()`` gathers, for every layer,
the prompt's K and V out of its paged pool into a contiguous
``[seq, kv_heads, head_dim]`` array; the decode instance's ``admit()`` then
computes one slot per prompt position from its own block table and writes the
gathered rows there. Section "布局转换" adds the TP difference: each side
keeps 1/T of the KV heads per card, so the gathered array is the prefill
cards' head ranges put side by side, and the decode side takes its own head
range out of it. With more cards than heads (the reading taken for T > H),
T/H consecutive cards hold the same head: the gather takes each head from the
first card of its group, and every card of a decode group receives its head.

Unlike the C loop nest, the gather here reads whole physical blocks (a
request's tokens are its blocks laid end to end in table order) and the
write uses pd.py's list of slots, so the two definitions share no indexing
expression.
"""
from __future__ import annotations

import numpy as np


def _shard_view(pool, num_layers, num_components, num_blocks, block, heads, head_dim):
    return pool.reshape(num_layers, num_components, num_blocks, block, heads, head_dim)


def gather_prefill(src_pools, layer, comp, block_ids, n, *, num_layers, num_components,
                   kv_heads, head_dim, src_tp, src_block, src_num_blocks):
    """pd.py ``prefill()`` gather of one layer/component: -> [n, kv_heads, head_dim]."""
    hp = kv_heads // src_tp if src_tp <= kv_heads else 1
    group = src_tp // kv_heads if src_tp > kv_heads else 1      # cards holding one head
    per_card = []
    for card, pool in enumerate(src_pools):
        if card % group:
            continue                       # a further copy of a head already gathered
        v = _shard_view(pool, num_layers, num_components, src_num_blocks, src_block, hp,
                        head_dim)
        blocks = v[layer, comp][np.asarray(block_ids, dtype=np.int64)]   # [nb, Bp, hp, D]
        per_card.append(blocks.reshape(-1, hp, head_dim)[:n])
    return np.concatenate(per_card, axis=1) if per_card else None


def admit_decode(dst_pools, layer, comp, block_ids, rows, *, num_layers, num_components,
                 kv_heads, head_dim, dst_tp, dst_block, dst_num_blocks):
    """pd.py ``admit()`` write of one layer/component from gathered ``rows``."""
    n = rows.shape[0]
    hd = kv_heads // dst_tp if dst_tp <= kv_heads else 1
    group = dst_tp // kv_heads if dst_tp > kv_heads else 1
    slots = np.array([block_ids[p // dst_block] * dst_block + p % dst_block
                      for p in range(n)], dtype=np.int64)
    for card, pool in enumerate(dst_pools):
        v = _shard_view(pool, num_layers, num_components, dst_num_blocks, dst_block, hd,
                        head_dim)
        flat = v[layer, comp].reshape(dst_num_blocks * dst_block, hd, head_dim)
        first = (card // group) * hd         # the card's first head
        flat[slots] = rows[:, first:first + hd, :]


def relayout(src_pools, dst_pools, *, num_layers, num_components, kv_heads, head_dim,
             elem_bytes, src_tp, dst_tp, src_block, dst_block, src_num_blocks,
             dst_num_blocks, seq_lens, src_off, src_bt, dst_off, dst_bt,
             layer_begin=0, layer_end=None):
    """Both halves of pd.py for every request and layer, in place on ``dst_pools``.

    ``elem_bytes`` is implied by the arrays' dtype (raw bit patterns); it is
    accepted so that the call matches the C oracle's.
    """
    del elem_bytes
    if layer_end is None:
        layer_end = num_layers
    geo = dict(num_layers=num_layers, num_components=num_components, kv_heads=kv_heads,
               head_dim=head_dim)
    for r, n in enumerate(np.asarray(seq_lens).tolist()):
        if n == 0:
            continue
        sblocks = np.asarray(src_bt[src_off[r]:src_off[r + 1]])
        dblocks = np.asarray(dst_bt[dst_off[r]:dst_off[r + 1]]).tolist()
        nb = -(-n // src_block)
        for layer in range(layer_begin, layer_end):
            for comp in range(num_components):
                rows = gather_prefill(src_pools, layer, comp, sblocks[:nb], n, src_tp=src_tp,
                                      src_block=src_block, src_num_blocks=src_num_blocks,
                                      **geo)
                admit_decode(dst_pools, layer, comp, dblocks, rows, dst_tp=dst_tp,
                             dst_block=dst_block, dst_num_blocks=dst_num_blocks, **geo)
