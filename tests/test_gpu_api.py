"""GPU behaviour of the C ABI: errors are statuses, streams, graphs, repeated launches."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import run, to_device, to_host
from prefill_decode_paged_gb300 import KVRelayoutError, RelayoutPlan

pytestmark = pytest.mark.gpu


def _small():
    return wl.custom("api", 7, num_layers=4, num_components=2, kv_heads=8, head_dim=64,
                     elem_bytes=2, src_tp=4, dst_tp=2, src_block=16, dst_block=64,
                     seq_lens=[500, 3, 129])


def _ref(w, src_np):
    ref = w.dst_pools_numpy()
    oracle.relayout(src_np, ref, **w.geometry())
    return ref


def test_bad_calls_return_statuses_and_leave_the_context_usable():
    import torch
    w = _small()
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        for bad in (-1, w.num_layers, 1 << 30):
            with pytest.raises(KVRelayoutError) as e:
                plan.run_layer(bad)
            assert e.value.name == "KVR_ERR_LAYER_RANGE"
    g = w.geometry()
    g["dst_bt"] = w.dst_bt.copy()
    g["dst_bt"][1] = g["dst_bt"][0]
    with pytest.raises(KVRelayoutError) as e:
        RelayoutPlan(src, dst, **g)
    assert e.value.name == "KVR_ERR_DST_ALIAS"
    with pytest.raises(KVRelayoutError) as e:
        RelayoutPlan(src, [dst[0], dst[0]], **w.geometry())
    assert e.value.name == "KVR_ERR_POOL_OVERLAP"
    misaligned = [src[0].data_ptr() + 8] + [t.data_ptr() for t in src[1:]]
    with pytest.raises(KVRelayoutError) as e:
        RelayoutPlan(misaligned, dst, **w.geometry())
    assert e.value.name == "KVR_ERR_ALIGNMENT"
    run(w, src, dst)
    for a, b in zip(_ref(w, src_np), to_host(dst, w)):
        np.testing.assert_array_equal(b, a)


def test_per_layer_on_a_side_stream_in_reverse_order():
    import torch
    w = _small()
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        with torch.cuda.stream(side):
            for layer in reversed(range(w.num_layers)):
                plan.run_layer(layer)            # binding default: the current (side) stream
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
    for a, b in zip(_ref(w, src_np), to_host(dst, w)):
        np.testing.assert_array_equal(b, a)


def test_layer_launch_ordered_after_the_producer_kernel():
    """The prefill side writes a layer with an ordinary kernel, the relayout of that
    layer follows on the same stream: it must see the new values."""
    import torch
    w = _small()
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        for layer in range(w.num_layers):
            for t in src:
                t[layer].bitwise_not_()          # "compute" layer l on the prefill side
            plan.run_layer(layer)
        torch.cuda.synchronize()
    flipped = [~a for a in src_np]
    for a, b in zip(_ref(w, flipped), to_host(dst, w)):
        np.testing.assert_array_equal(b, a)


def test_chained_hand_offs_see_the_previous_launchs_writes():
    """A's decode pools are B's prefill pools; per-layer launches alternate A, B on one
    stream. Each launch lets the next one start early and prefetch its prefill rows
    into L2 while the previous launch may still be writing them; B must still read
    what A wrote (the oracle applied twice), layer after layer."""
    import dataclasses
    import torch
    a = wl.custom("chainA", 21, num_layers=4, num_components=2, kv_heads=8, head_dim=128,
                  elem_bytes=2, src_tp=2, dst_tp=4, src_block=16, dst_block=32,
                  seq_lens=[300, 77, 1])
    # B reads A's decode side: same shards, blocks and tables; writes 1 shard of 64-token blocks
    b0 = wl.custom("chainB", 22, num_layers=4, num_components=2, kv_heads=8, head_dim=128,
                   elem_bytes=2, src_tp=4, dst_tp=1, src_block=32, dst_block=64,
                   seq_lens=[300, 77, 1])
    b = dataclasses.replace(b0, src_num_blocks=a.dst_num_blocks, src_off=a.dst_off,
                            src_bt=a.dst_bt)
    src_np = a.src_pools_numpy()
    mid_ref = _ref(a, src_np)
    want = _ref(b, mid_ref)
    src = to_device(src_np, 2)
    for _ in range(3):
        mid = to_device(a.dst_pools_numpy(), 2)
        dst = to_device(b.dst_pools_numpy(), 2)
        with RelayoutPlan(src, mid, **a.geometry()) as pa, \
                RelayoutPlan(mid, dst, **b.geometry()) as pb:
            for layer in range(a.num_layers):
                pa.run_layer(layer)
                pb.run_layer(layer)
            torch.cuda.synchronize()
        for x, y in zip(want, to_host(dst, b)):
            np.testing.assert_array_equal(y, x)


def test_captured_in_a_cuda_graph_and_replayed():
    import torch
    w = _small()
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    plan = RelayoutPlan(src, dst, **w.geometry())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for layer in range(w.num_layers):
            plan.run_layer(layer)
    for t in dst:
        t.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(_ref(w, src_np), to_host(dst, w)):
        np.testing.assert_array_equal(b, a)
    plan.close()


def test_empty_batch_and_repeated_launches():
    import torch
    w = wl.custom("z", 8, num_layers=2, num_components=2, kv_heads=2, head_dim=8, elem_bytes=2,
                  src_tp=1, dst_tp=1, src_block=16, dst_block=32, seq_lens=[0, 0])
    src = to_device(w.src_pools_numpy(), 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        assert plan.bytes_read == plan.bytes_written == 0
        plan.run_all()
        plan.run_layer(1)
        torch.cuda.synchronize()
    assert all(bool((t == -1).all()) for t in dst)
    w = _small()
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        for _ in range(3):
            plan.run_all()
        torch.cuda.synchronize()
    for a, b in zip(_ref(w, src_np), to_host(dst, w)):
        np.testing.assert_array_equal(b, a)


def _pinned_like(tensors):
    import torch
    out = []
    for t in tensors:
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        out.append(h)
    return out


def test_pools_in_pinned_host_memory():
    """Prefill and/or decode pools in pinned host memory: the kernel reaches them
    directly (no staging copy) and the bytes are the oracle's."""
    import torch
    w = _small()
    src_np = w.src_pools_numpy()
    ref = _ref(w, src_np)
    dev_src = to_device(src_np, 2)
    host_src = _pinned_like(dev_src)
    for src in (host_src, dev_src):
        for host_dst in (True, False):
            dst = to_device(w.dst_pools_numpy(), 2)
            if host_dst:
                dst = _pinned_like(dst)
            if src is dev_src and not host_dst:
                continue
            with RelayoutPlan(src, dst, **w.geometry()) as plan:
                plan.run_all()
                torch.cuda.synchronize()
            for a, t in zip(ref, dst):
                np.testing.assert_array_equal(t.cpu().numpy().view(np.uint16), a)


def test_pools_the_gpu_cannot_reach_are_refused():
    import torch
    from prefill_decode_paged_gb300 import relayout_all_prealloc
    w = _small()
    src = to_device(w.src_pools_numpy(), 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    pageable = [np.zeros(w.src_shape(), dtype=np.int16) for _ in range(w.src_tp)]
    bad_src = [a.ctypes.data // 256 * 256 + 256 for a in pageable]   # 16-B aligned, pageable
    with pytest.raises(KVRelayoutError) as e:
        RelayoutPlan(bad_src, dst, **w.geometry())
    assert e.value.name == "KVR_ERR_POOL_ADDRESS"
    with pytest.raises(KVRelayoutError) as e:
        relayout_all_prealloc(src, [a.ctypes.data // 256 * 256 + 256 for a in
                                    [np.zeros(w.dst_shape(), np.int16) for _ in range(2)]],
                              **w.geometry())
    assert e.value.name == "KVR_ERR_POOL_ADDRESS"
    torch.cuda.synchronize()
    assert all(bool((t == -1).all()) for t in dst)


def test_launch_shape_fills_the_gpu_per_layer():
    """128 tiles of 64 decode tokens per layer: a per-layer launch splits them to cover
    every SM; a whole-prompt launch holds every (layer, tile) task. The relayout
    matches the oracle in both modes."""
    import torch
    w = wl.custom("shape", 9, num_layers=4, num_components=2, kv_heads=8, head_dim=128,
                  elem_bytes=2, src_tp=2, dst_tp=1, src_block=16, dst_block=64,
                  seq_lens=[2048] * 4)
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ref = _ref(w, src_np)
    for mode in ("all", "layer"):
        dst = to_device(w.dst_pools_numpy(), 2)
        with RelayoutPlan(src, dst, **w.geometry()) as plan:
            grid_all, grid_layer, tile = plan.launch_shape
            if mode == "all":
                plan.run_all()
            else:
                for layer in range(w.num_layers):
                    plan.run_layer(layer)
            torch.cuda.synchronize()
        for a, b in zip(ref, to_host(dst, w)):
            np.testing.assert_array_equal(b, a)
    assert tile == 64
    items = 4 * 2048 // 64
    assert grid_layer % items == 0 and grid_layer >= sms
    assert grid_all % (items * w.num_layers) == 0


@pytest.mark.parametrize("groups", [[4], [1, 3], [2, 2], [3, 1], [1, 2, 1]])
def test_layer_ranges_match_the_oracle(groups):
    """kv_relayout_layers over any split of the layers equals the whole relayout."""
    import torch
    w = _small()
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        first = 0
        for count in groups:
            plan.run_layers(first, count)
            first += count
        torch.cuda.synchronize()
    for a, b in zip(_ref(w, src_np), to_host(dst, w)):
        np.testing.assert_array_equal(b, a)


def test_layer_range_errors_are_statuses():
    import torch
    w = _small()
    src = to_device(w.src_pools_numpy(), 2)
    dst = to_device(w.dst_pools_numpy(), 2)
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        for first, count in ((-1, 1), (0, 0), (3, 2), (4, 1), (0, 5)):
            with pytest.raises(KVRelayoutError) as e:
                plan.run_layers(first, count)
            assert e.value.name == "KVR_ERR_LAYER_RANGE"
        plan.run_layers(0, 4)
        torch.cuda.synchronize()


def test_no_wait_launches_after_hand_off_launches():
    """Back-to-back single-layer launches where every launch but the first passes
    KVR_LAUNCH_NO_WAIT (each follows another hand-off launch of the same plan; all
    prefill rows were ready before the first): same bytes as one whole launch,
    eager and captured in a CUDA graph."""
    import torch
    w = wl.custom("nw", 13, num_layers=6, num_components=2, kv_heads=8, head_dim=128,
                  elem_bytes=2, src_tp=4, dst_tp=8, src_block=16, dst_block=32,
                  seq_lens=[1500, 77, 640])
    src_np = w.src_pools_numpy()
    src = to_device(src_np, 2)
    ref = _ref(w, src_np)
    for graph in (False, True):
        dst = to_device(w.dst_pools_numpy(), 2)
        with RelayoutPlan(src, dst, **w.geometry()) as plan:
            def launches():
                for layer in range(w.num_layers):
                    plan.run_layers(layer, 1, wait_for_previous=layer == 0)
            if graph:
                g = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream()
                cap.wait_stream(torch.cuda.current_stream())
                with torch.cuda.graph(g, stream=cap):
                    launches()
                torch.cuda.current_stream().wait_stream(cap)
                g.replay()
            else:
                launches()
            # work queued right after the chain on the same stream sees every launch's
            # writes: the copies below run before any host synchronization
            snap = [t.clone() for t in dst]
            torch.cuda.synchronize()
        for a, b, c in zip(ref, to_host(dst, w), to_host(snap, w)):
            np.testing.assert_array_equal(b, a)
            np.testing.assert_array_equal(c, a)
    with RelayoutPlan(src, to_device(w.dst_pools_numpy(), 2), **w.geometry()) as plan:
        st = plan._handle()
        from prefill_decode_paged_gb300.kv_relayout import library
        assert library().kv_relayout_layers_ex(st, 0, 1, 2, None) == -1   # unknown flag


def test_plain_c_client_on_the_gpu():
    """A C99 program (kv_relayout.h, cudaMalloc, no Python in the loop) plans and runs
    whole-prompt, per-layer and layer-range launches; every decode byte matches the
    C oracle."""
    import subprocess
    from test_host_abi import build_abi_client
    exe = build_abi_client()
    out = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert "gpu: ok" in out.stdout
