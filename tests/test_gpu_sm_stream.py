"""The relayout on streams limited to a number of SMs (green contexts)."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import to_device, to_host
from prefill_decode_paged_gb300 import KVRelayoutError, RelayoutPlan, SmStream

pytestmark = pytest.mark.gpu


def test_relayout_on_sm_limited_streams_is_exact_and_slower_on_few_sms():
    import torch
    total = torch.cuda.get_device_properties(0).multi_processor_count
    w = wl.custom("sms", 17, num_layers=4, num_components=2, kv_heads=8, head_dim=128,
                  elem_bytes=2, src_tp=4, dst_tp=8, src_block=16, dst_block=32,
                  seq_lens=[4096, 1000], values="randn")
    src_np = w.src_pools_numpy()
    ref = w.dst_pools_numpy()
    oracle.relayout(src_np, ref, **w.geometry())
    src = to_device(src_np, 2)
    times = {}
    for want in (8, 24, total):
        with SmStream(want) as s:
            assert s.sms >= want and (want == total or s.sms % 8 == 0)
            dst = to_device(w.dst_pools_numpy(), 2)
            with RelayoutPlan(src, dst, **w.geometry()) as plan:
                ext = torch.cuda.ExternalStream(s.handle)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                plan.run_all(s.handle)
                ext.synchronize()
                for a, b in zip(ref, to_host(dst, w)):
                    np.testing.assert_array_equal(b, a)
                ev[0].record(ext)
                for _ in range(20):
                    plan.run_all(s.handle)
                ev[1].record(ext)
                ext.synchronize()
                times[want] = ev[0].elapsed_time(ev[1]) / 20
    assert times[8] > 2.0 * times[total], times


def test_sm_stream_rejects_more_sms_than_the_gpu_has():
    import torch
    total = torch.cuda.get_device_properties(0).multi_processor_count
    with pytest.raises(KVRelayoutError) as e:
        SmStream(total + 1)
    assert e.value.name == "KVR_ERR_INVALID_ARG"


def test_layer_ranges_on_an_sm_limited_stream():
    """Launches on a green-context stream are shaped for its SMs; the bytes are the
    same as on the whole GPU."""
    import torch
    w = wl.custom("smr", 18, num_layers=5, num_components=2, kv_heads=8, head_dim=128,
                  elem_bytes=2, src_tp=2, dst_tp=1, src_block=16, dst_block=256,
                  seq_lens=[2000, 300])
    src_np = w.src_pools_numpy()
    ref = w.dst_pools_numpy()
    oracle.relayout(src_np, ref, **w.geometry())
    src = to_device(src_np, 2)
    with SmStream(16) as s:
        ext = torch.cuda.ExternalStream(s.handle)
        for split in ([5], [2, 3], [1, 4]):
            dst = to_device(w.dst_pools_numpy(), 2)
            with RelayoutPlan(src, dst, **w.geometry()) as plan:
                first = 0
                for count in split:
                    if count == w.num_layers:
                        plan.run_all(s.handle)
                    else:
                        plan.run_layers(first, count, s.handle)
                    first += count
                ext.synchronize()
            for a, b in zip(ref, to_host(dst, w)):
                np.testing.assert_array_equal(b, a)
