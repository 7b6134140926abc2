"""Seeded random geometries for the fuzz tests (CPU emulator and GPU parity).

Every draw is a valid hand-off: each TP degree divides H or (about one side in
four) is a multiple of it, so heads are replicated; rows of a whole number of
16-byte units, lengths from 0 to a few blocks of either side (ragged
tails on both), optional shared prefill prefix, pools with slack.
"""
import numpy as np

import workloads as wl


def random_workload(seed: int, max_tokens: int = 700, elem_bytes=None, head_dim_multiple=1):
    """``elem_bytes`` fixes the element width; ``head_dim_multiple`` restricts head_dim
    (16 for a converting relayout, whose units are 16 elements)."""
    rng = np.random.default_rng([seed, 77])
    es = int(rng.choice([1, 2, 4])) if elem_bytes is None else int(elem_bytes)
    tps = [1, 2, 3, 4, 6, 8]
    H = int(rng.choice([1, 2, 4, 6, 8, 12, 16]))
    src_tp = int(rng.choice([t for t in tps if H % t == 0]))
    dst_tp = int(rng.choice([t for t in tps if H % t == 0]))
    # a second stream decides replication, so the draws below stay those of the seed
    rep = np.random.default_rng([seed, 78])
    multiples = [m for m in (2, 4, 8, 16) if H * m <= 16]
    if multiples and rep.random() < 0.25:
        src_tp = H * int(rep.choice(multiples))
    if multiples and rep.random() < 0.25:
        dst_tp = H * int(rep.choice(multiples))
    d_choices = [d for d in (8, 16, 24, 32, 64, 72, 128, 576)
                 if (d * es) % 16 == 0 and d % head_dim_multiple == 0]
    D = int(rng.choice(d_choices))
    C = int(rng.choice([1, 2]))
    L = int(rng.integers(1, 5))
    bp = int(rng.choice([1, 3, 8, 16, 32, 64]))
    bd = int(rng.choice([1, 5, 16, 32, 64, 256]))
    R = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(0, max_tokens, size=R)]
    if rng.random() < 0.3:
        lens[int(rng.integers(0, R))] = 0
    shared = int(rng.integers(0, 3)) if bp > 1 and R > 1 else 0
    return wl.custom(f"fz{seed}", 1000 + seed, num_layers=L, num_components=C, kv_heads=H,
                     head_dim=D, elem_bytes=es, src_tp=src_tp, dst_tp=dst_tp, src_block=bp,
                     dst_block=bd, seq_lens=lens, shared_prefix=shared)
