"""kv_relayout_all_prealloc: the whole-prompt relayout for callers that cannot allocate.

Some callers cannot call cudaMalloc while they hand KV over: an engine that
has already carved its HBM into KV block pools has no room for one more
buffer, and a latency-critical loop cannot pay the device-wide
synchronization of cudaMalloc/cudaFree. This entry point keeps its work list
in a fixed device array inside the library instead of a per-plan allocation.
Every call reuses that array, which still holds the previous call's work
list, so the tests below call it several times in a row, with work lists of
different sizes, and require the same bytes as the allocating path
(kv_relayout_plan + kv_relayout_all), bit for bit: this is a bit copy, so the
tolerance is zero.

This file is collected last on purpose.
"""
import pytest

import workloads as wl
from prefill_decode_paged_gb300 import KVRelayoutError, RelayoutPlan, relayout_all_prealloc
from prefill_decode_paged_gb300.kv_relayout import PREALLOC_SCRATCH_BYTES

pytestmark = pytest.mark.gpu


def _both_paths(w):
    import torch
    src = w.src_pools_torch("cuda")
    ref = w.dst_pools_torch("cuda")
    got = w.dst_pools_torch("cuda")
    with RelayoutPlan(src, ref, **w.geometry()) as plan:
        plan.run_all()
        relayout_all_prealloc(src, got, **w.geometry())
        torch.cuda.synchronize()
    for s, (a, b) in enumerate(zip(ref, got)):
        assert torch.equal(a, b), f"{w.name}: shard {s} differs from the allocating path"
    # the allocating path itself moved the prompt (the comparison is not vacuous)
    assert any(bool((t != -1).any()) for t in ref)


def test_calls_in_a_row_match_the_allocating_entry_point():
    big = wl.custom("prealloc_big", 31, num_layers=3, num_components=2, kv_heads=8,
                    head_dim=64, elem_bytes=2, src_tp=4, dst_tp=8, src_block=16,
                    dst_block=32, seq_lens=[3000, 17, 1200], values="randn")
    small = wl.custom("prealloc_small", 32, num_layers=2, num_components=1, kv_heads=1,
                      head_dim=576, elem_bytes=2, src_tp=1, dst_tp=1, src_block=64,
                      dst_block=16, seq_lens=[300, 65], values="randn")
    ragged = wl.custom("prealloc_ragged", 33, num_layers=2, num_components=2, kv_heads=6,
                       head_dim=8, elem_bytes=2, src_tp=3, dst_tp=2, src_block=3,
                       dst_block=5, seq_lens=[40, 0, 17, 1])
    # heads replicated over TP (an MLA latent on 2 prefill and 4 decode shards)
    replicated = wl.custom("prealloc_replicated", 35, num_layers=2, num_components=1,
                           kv_heads=1, head_dim=576, elem_bytes=2, src_tp=2, dst_tp=4,
                           src_block=64, dst_block=16, seq_lens=[300, 65], values="randn")
    # the second call's work list is shorter than the first's, so stale entries of
    # the first call are still in the array behind it; the third call grows again
    for w in (big, small, ragged, big, replicated):
        _both_paths(w)


def test_work_list_beyond_the_scratch_is_rejected_before_any_work():
    import torch
    # one-token blocks on both sides: 4 + 4 bytes of block ids per token
    n = PREALLOC_SCRATCH_BYTES // 8 + 1000
    w = wl.custom("prealloc_too_big", 34, num_layers=1, num_components=1, kv_heads=1,
                  head_dim=8, elem_bytes=2, src_tp=1, dst_tp=1, src_block=1, dst_block=1,
                  seq_lens=[n], values="randn")
    src = w.src_pools_torch("cuda")
    dst = w.dst_pools_torch("cuda")
    with pytest.raises(KVRelayoutError) as e:
        relayout_all_prealloc(src, dst, **w.geometry())
    assert e.value.name == "KVR_ERR_SCRATCH_LIMIT"
    torch.cuda.synchronize()
    assert all(bool((t == -1).all()) for t in dst)
    # the allocating path still handles it
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        plan.run_all()
        torch.cuda.synchronize()
    assert int((dst[0] != -1).sum()) == n * 8
