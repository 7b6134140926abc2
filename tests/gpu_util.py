"""Helpers for the GPU parity tests: move seeded pools to the device and back, run plans."""
from __future__ import annotations

import dataclasses

import numpy as np

_NP_VIEW = {1: np.uint8, 2: np.int16, 4: np.int32}


def torch_dtype(es):
    import torch
    return {1: torch.uint8, 2: torch.int16, 4: torch.int32}[es]


def to_device(arrays, es):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(a).view(_NP_VIEW[es])).cuda() for a in arrays]


def to_host(tensors, w):
    return [t.cpu().numpy().view(w.int_dtype()) for t in tensors]


def run(w, src, dst, mode="all", stream=None):
    """Plan + launch through the C ABI, then wait for the device."""
    import torch
    from prefill_decode_paged_gb300 import RelayoutPlan
    with RelayoutPlan(src, dst, **w.geometry()) as plan:
        if mode == "all":
            plan.run_all(stream)
        else:
            for layer in range(w.num_layers):
                plan.run_layer(layer, stream)
        torch.cuda.synchronize()


def oracle_layer(w, src_dev, layer):
    """The oracle's result for one layer, computed from that layer's prefill slices."""
    import oracle
    w1 = dataclasses.replace(w, num_layers=1)
    src = [np.ascontiguousarray(t[layer:layer + 1].cpu().numpy().view(w.int_dtype()))
           for t in src_dev]
    dst = w1.dst_pools_numpy()
    oracle.relayout(src, dst, **w1.geometry())
    return dst
