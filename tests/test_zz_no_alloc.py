"""kv_relayout_all_prealloc: the whole-prompt relayout for callers that cannot allocate.

Some callers cannot call cudaMalloc while they hand KV over: an engine that
has already carved its HBM into KV block pools has no room for one more
buffer, and a latency-critical loop cannot pay the device-wide
synchronization of cudaMalloc/cudaFree. This entry point keeps its work list
in a fixed device array inside the library instead of a per-plan allocation.
Every call reuses that array, which still holds the previous call's work
list, so the tests below call it several times in a row, with work lists of
different sizes, and require the same bytes as the allocating path
(kv_relayout_plan + kv_relayout_all) and as the CPU oracle, bit for bit: this
is a bit copy, so the tolerance is zero.

This file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import to_device, to_host
from prefill_decode_paged_gb300 import KVRelayoutError, RelayoutPlan, relayout_all_prealloc
from prefill_decode_paged_gb300.kv_relayout import PREALLOC_SCRATCH_BYTES

pytestmark = pytest.mark.gpu

BIG = lambda: wl.custom("prealloc_big", 31, num_layers=3, num_components=2, kv_heads=8,  # noqa
                        head_dim=64, elem_bytes=2, src_tp=4, dst_tp=8, src_block=16,
                        dst_block=32, seq_lens=[3000, 17, 1200], values="randn")
SMALL = lambda: wl.custom("prealloc_small", 32, num_layers=2, num_components=1,  # noqa
                          kv_heads=1, head_dim=576, elem_bytes=2, src_tp=1, dst_tp=1,
                          src_block=64, dst_block=16, seq_lens=[300, 65], values="randn")
# partial blocks on both sides, an empty prompt, a TP3 -> TP2 merge of 6 heads
RAGGED = lambda: wl.custom("prealloc_ragged", 33, num_layers=2, num_components=2,  # noqa
                           kv_heads=6, head_dim=8, elem_bytes=2, src_tp=3, dst_tp=2,
                           src_block=3, dst_block=5, seq_lens=[40, 0, 17, 1])
# heads replicated over TP (an MLA latent on 2 prefill and 4 decode shards)
REPLICATED = lambda: wl.custom("prealloc_replicated", 35, num_layers=2,  # noqa
                               num_components=1, kv_heads=1, head_dim=576, elem_bytes=2,
                               src_tp=2, dst_tp=4, src_block=64, dst_block=16,
                               seq_lens=[300, 65], values="randn")


def _oracle(w, src_np):
    ref = w.dst_pools_numpy()
    oracle.relayout(src_np, ref, **w.geometry())
    return ref


def _both_paths(w):
    import torch
    src_np = w.src_pools_numpy()
    src = to_device(src_np, w.elem_bytes)
    ref = w.dst_pools_torch("cuda")
    got = w.dst_pools_torch("cuda")
    with RelayoutPlan(src, ref, **w.geometry()) as plan:
        plan.run_all()
        relayout_all_prealloc(src, got, **w.geometry())
        torch.cuda.synchronize()
    for s, (a, b) in enumerate(zip(ref, got)):
        assert torch.equal(a, b), f"{w.name}: shard {s} differs from the allocating path"
    # both equal the CPU oracle, element by element (sentinel bytes included)
    for s, (a, b) in enumerate(zip(_oracle(w, src_np), to_host(got, w))):
        assert np.array_equal(a, b), f"{w.name}: shard {s} differs from the oracle"
    # the prompt was moved (the comparison is not vacuous)
    assert any(bool((t != -1).any()) for t in ref) or not int(w.seq_lens.sum())


def test_calls_in_a_row_match_the_allocating_entry_point_and_the_oracle():
    # the second call's work list is shorter than the first's, so stale entries of
    # the first call are still in the array behind it; the fourth call grows again
    for make in (BIG, SMALL, RAGGED, BIG, REPLICATED):
        _both_paths(make())


def test_calls_queued_back_to_back_on_one_stream():
    """Several calls with different work lists queued on one stream with no host
    synchronization between them, the first right after a per-layer launch that lets
    its successor start early (programmatic dependent launch): each call's copy of its
    work list must wait for the kernel before it, which still reads the previous list."""
    import torch
    stream = torch.cuda.Stream()
    cases = [make() for make in (BIG, RAGGED, REPLICATED, SMALL)]
    srcs_np = [w.src_pools_numpy() for w in cases]
    srcs = [to_device(s, w.elem_bytes) for s, w in zip(srcs_np, cases)]
    dsts = [w.dst_pools_torch("cuda") for w in cases]
    first = cases[0]
    layer_dst = first.dst_pools_torch("cuda")
    torch.cuda.synchronize()
    with RelayoutPlan(srcs[0], layer_dst, **first.geometry()) as plan:
        plan.run_layer(0, stream)
        for w, src, dst in zip(cases, srcs, dsts):
            relayout_all_prealloc(src, dst, stream, **w.geometry())
        stream.synchronize()
    for w, src_np, dst in zip(cases, srcs_np, dsts):
        for s, (a, b) in enumerate(zip(_oracle(w, src_np), to_host(dst, w))):
            assert np.array_equal(a, b), f"{w.name}: shard {s} differs from the oracle"
    # the per-layer launch moved layer 0 only
    ref = _oracle(first, srcs_np[0])
    for a, b in zip(ref, to_host(layer_dst, first)):
        assert np.array_equal(a[:1], b[:1]) and bool((b[1:] == 0xFFFF).all())


def test_refused_while_the_stream_is_captured():
    """The call copies its tables from host memory it frees on return, so it enqueues
    nothing on a stream under capture; the capture stays valid."""
    import torch
    w = SMALL()
    src = to_device(w.src_pools_numpy(), w.elem_bytes)
    dst = w.dst_pools_torch("cuda")
    relayout_all_prealloc(src, dst, **w.geometry())     # first call: before any capture
    torch.cuda.synchronize()
    graph_dst = w.dst_pools_torch("cuda")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with RelayoutPlan(src, graph_dst, **w.geometry()) as plan:
        with torch.cuda.graph(g, stream=side):
            with pytest.raises(KVRelayoutError) as e:
                relayout_all_prealloc(src, graph_dst, **w.geometry())
            plan.run_all()
        assert e.value.name == "KVR_ERR_UNSUPPORTED"
        torch.cuda.synchronize()
        assert all(bool((t == -1).all()) for t in graph_dst)
        g.replay()
        torch.cuda.synchronize()
    for a, b in zip(dst, graph_dst):
        assert torch.equal(a, b)
    del g


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


def test_call_on_an_sm_limited_stream_matches_the_oracle():
    """On a stream limited to a few SMs (a green context) the call shapes its grid for
    that stream's SMs, as the allocating path does; the bytes are the oracle's."""
    import torch
    from prefill_decode_paged_gb300 import SmStream
    w = BIG()
    src_np = w.src_pools_numpy()
    src = to_device(src_np, w.elem_bytes)
    dst = w.dst_pools_torch("cuda")
    try:
        s = SmStream(16)
    except KVRelayoutError as e:
        pytest.skip(f"no green contexts here: {e.name}")
    with s:
        relayout_all_prealloc(src, dst, s.handle, **w.geometry())
        torch.cuda.ExternalStream(s.handle).synchronize()
    for k, (a, b) in enumerate(zip(_oracle(w, src_np), to_host(dst, w))):
        assert np.array_equal(a, b), f"shard {k} differs from the oracle"
