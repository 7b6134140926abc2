"""Pins of the oracle's dtype-converting relayout (BF16 <-> FP8 E4M3).

The codecs are pinned to values the OCP 8-bit floating point specification
fixes for E4M3 (field layout, 448 as the largest finite value, 2^-9 as the
smallest subnormal, S.1111.111 as NaN) and to torch's CPU casts (a library
routine: nearest, ties to even) on every value where those casts are defined
the same way (finite, in range). The converting relayout's placement is
pinned to the already-pinned copy relayout: with power-of-two scales the
conversion of each element is exact, so the converted pools must equal a
plain relayout of pre-converted pools.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

F8 = torch.float8_e4m3fn


def _torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(F8).float().numpy()


# -- codecs --------------------------------------------------------------------

def test_e4m3_decode_fixed_points(oracle_lib):
    d = oracle.e4m3_decode(np.arange(256, dtype=np.uint8), lib=oracle_lib)
    assert d[0x00] == 0.0 and np.signbit(d[0x80]) and d[0x80] == 0.0
    assert d[0x01] == 2.0 ** -9 and d[0x07] == 7 * 2.0 ** -9     # subnormals
    assert d[0x08] == 2.0 ** -6                                  # smallest normal
    assert d[0x38] == 1.0 and d[0x40] == 2.0 and d[0x3C] == 1.5
    assert d[0x7E] == 448.0 and d[0xFE] == -448.0                # largest finite
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])               # the only NaNs
    assert np.isnan(d).sum() == 2
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0)                              # codes are ordered
    np.testing.assert_array_equal(d[0x80:0xFF], -pos)


def test_e4m3_decode_matches_torch(oracle_lib):
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8), lib=oracle_lib)
    ref = _torch_e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_e4m3_round_trip(oracle_lib):
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes, lib=oracle_lib), lib=oracle_lib)
    np.testing.assert_array_equal(back, codes)


def test_e4m3_encode_matches_torch_in_range(oracle_lib):
    v = _torch_e4m3_values()[:0x7F].astype(np.float64)
    mids = (v[:-1] + v[1:]) / 2                                   # exact ties
    rng = np.random.default_rng(5)
    x = np.concatenate([
        mids, -mids,
        np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
        np.nextafter(mids.astype(np.float32), np.float32(-np.inf)),
        rng.uniform(-448, 448, 20000),
        rng.standard_normal(20000) * 0.05,
        np.ldexp(rng.uniform(-1, 1, 5000), -8),                   # subnormal range
        [0.0, -0.0, 448.0, -448.0],
    ]).astype(np.float32)
    ours = oracle.e4m3_encode(x, lib=oracle_lib)
    ref = torch.from_numpy(x).to(F8).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_encode_saturates_and_keeps_nan(oracle_lib):
    x = np.array([449.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf, np.nan, -np.nan],
                 dtype=np.float32)
    x[-1] = -np.abs(x[-1])
    got = oracle.e4m3_encode(x, lib=oracle_lib)
    assert list(got[:5]) == [0x7E] * 5
    assert list(got[5:7]) == [0xFE] * 2
    assert got[7] == 0x7F and got[8] == 0xFF


def test_bf16_encode_matches_torch(oracle_lib):
    rng = np.random.default_rng(6)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    # force many exact ties (low half 0x8000) with both parities of the kept bit
    bits[:50000] = (bits[:50000] & 0xFFFF0000) | 0x8000
    x = bits.view(np.float32)
    x = np.concatenate([x, np.float32([3.3895e38, 3.4e38, -3.4e38, 1e-40, -1e-45, 0.0, -0.0,
                                       np.inf, -np.inf])])
    finite_or_inf = ~np.isnan(x)
    ours = oracle.bf16_encode(x, lib=oracle_lib)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours[finite_or_inf], ref[finite_or_inf])
    nanv = ours[~finite_or_inf]
    assert np.all((nanv & 0x7FFF) == 0x7FC0)


# -- converting relayout: placement and scales -----------------------------------------

def _geometry(w):
    g = w.geometry()
    g.pop("elem_bytes")
    return g


def _conv_workload(seed, **kw):
    base = dict(num_layers=3, num_components=2, kv_heads=8, head_dim=16, elem_bytes=2,
                src_tp=4, dst_tp=2, src_block=16, dst_block=64, seq_lens=[300, 1, 77, 0])
    base.update(kw)
    return wl.custom("conv", seed, **base)


def _head_of_each_src_element(w):
    """Global head index of every element of each prefill shard (by layout meaning)."""
    hl = w.kv_heads // w.src_tp
    out = []
    for s in range(w.src_tp):
        h = s * hl + np.arange(hl)
        out.append(np.broadcast_to(h[None, None, None, None, :, None], w.src_shape()))
    return out


def _pow2_scales(rng, w, per_head):
    n = w.num_layers * w.num_components * (w.kv_heads if per_head else 1)
    return np.ldexp(np.ones(n, np.float32), rng.integers(-3, 4, n)).astype(np.float32)


def _scale_of_src(w, scales, per_head):
    """Per-element scale for each prefill shard."""
    L, C, H = w.num_layers, w.num_components, w.kv_heads
    heads = _head_of_each_src_element(w)
    out = []
    for s in range(w.src_tp):
        l = np.arange(L)[:, None, None, None, None, None]
        c = np.arange(C)[None, :, None, None, None, None]
        idx = ((l * C + c) * H + heads[s]) if per_head else (l * C + c + 0 * heads[s])
        out.append(scales[idx])
    return out


@pytest.mark.parametrize("per_head", [0, 1])
def test_quantize_placement_reduces_to_a_copy_of_codes(oracle_lib, per_head):
    rng = np.random.default_rng(10 + per_head)
    w = _conv_workload(12 + per_head)
    scales = _pow2_scales(rng, w, per_head)
    per_elem = _scale_of_src(w, scales, per_head)
    # source values: random E4M3-representable values times the element's scale (exact)
    vals = _torch_e4m3_values()
    finite_codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    src, codes = [], []
    for s in range(w.src_tp):
        c = rng.choice(finite_codes, size=w.src_shape()).astype(np.uint8)
        x = vals[c].astype(np.float32) * per_elem[s]
        xb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float()
                              .numpy(), x)                         # exact in bf16
        src.append(xb)
        codes.append(c)
    got = [np.full(w.dst_shape(), 0xFF, np.uint8) for _ in range(w.dst_tp)]
    oracle.relayout_convert(src, got, src_dtype=oracle.BF16, dst_dtype=oracle.E4M3,
                            per_head=per_head, scales=scales, lib=oracle_lib, **_geometry(w))
    want = [np.full(w.dst_shape(), 0xFF, np.uint8) for _ in range(w.dst_tp)]
    oracle.relayout(codes, want, lib=oracle_lib, **dict(w.geometry(), elem_bytes=1))
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("per_head", [0, 1])
def test_dequantize_placement_reduces_to_a_copy_of_values(oracle_lib, per_head):
    rng = np.random.default_rng(20 + per_head)
    w = _conv_workload(22 + per_head, elem_bytes=1, src_tp=2, dst_tp=4, src_block=64,
                       dst_block=16)
    scales = _pow2_scales(rng, w, per_head)
    per_elem = _scale_of_src(w, scales, per_head)
    vals = _torch_e4m3_values()
    finite_codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    src, pre = [], []
    for s in range(w.src_tp):
        c = rng.choice(finite_codes, size=w.src_shape()).astype(np.uint8)
        y = vals[c].astype(np.float32) * per_elem[s]                # exact in bf16
        src.append(c)
        pre.append(torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy()
                   .view(np.uint16))
    got = [np.full(w.dst_shape(), 0xFFFF, np.uint16) for _ in range(w.dst_tp)]
    oracle.relayout_convert(src, got, src_dtype=oracle.E4M3, dst_dtype=oracle.BF16,
                            per_head=per_head, scales=scales, lib=oracle_lib, **_geometry(w))
    want = [np.full(w.dst_shape(), 0xFFFF, np.uint16) for _ in range(w.dst_tp)]
    oracle.relayout(pre, want, lib=oracle_lib, **dict(w.geometry(), elem_bytes=2))
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)


def test_quantize_then_dequantize_stays_within_e4m3_precision(oracle_lib):
    rng = np.random.default_rng(30)
    w = _conv_workload(31, num_layers=2)
    scales = rng.uniform(0.01, 0.2, w.num_layers * w.num_components).astype(np.float32)
    src = w.src_pools_numpy()
    x = [torch.from_numpy(np.ascontiguousarray(
        (rng.standard_normal(w.src_shape()).astype(np.float32)))).to(torch.bfloat16)
        .view(torch.int16).numpy().view(np.uint16) for _ in src]
    q = [np.full(w.dst_shape(), 0xFF, np.uint8) for _ in range(w.dst_tp)]
    oracle.relayout_convert(x, q, src_dtype=oracle.BF16, dst_dtype=oracle.E4M3, per_head=0,
                            scales=scales, lib=oracle_lib, **_geometry(w))
    back_w = dataclasses.replace(w, src_tp=w.dst_tp, dst_tp=w.src_tp, src_block=w.dst_block,
                                 dst_block=w.src_block, src_num_blocks=w.dst_num_blocks,
                                 dst_num_blocks=w.src_num_blocks, src_off=w.dst_off,
                                 src_bt=w.dst_bt, dst_off=w.src_off, dst_bt=w.src_bt)
    back = [np.zeros(w.src_shape(), np.uint16) for _ in range(w.src_tp)]
    oracle.relayout_convert(q, back, src_dtype=oracle.E4M3, dst_dtype=oracle.BF16, per_head=0,
                            scales=scales, lib=oracle_lib, **_geometry(back_w))
    from kvcheck import covered_mask, full_mask
    cover = full_mask(w.src_shape(), covered_mask(w.src_shape(), w.src_off, w.src_bt,
                                                  w.seq_lens))
    L, C = w.num_layers, w.num_components
    s_el = np.broadcast_to(scales.reshape(L, C, 1, 1, 1, 1), w.src_shape())
    for a, b in zip(x, back):
        xa = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float().numpy()
        xb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
        m = cover & (np.abs(xa) / s_el >= 2.0 ** -6) & (np.abs(xa) / s_el <= 448)
        rel = np.abs(xb[m] - xa[m]) / np.abs(xa[m])
        assert m.sum() > 1000 and rel.max() <= 2.0 ** -4 + 2.0 ** -7
        assert np.all(b[~cover] == 0)


def test_nan_keeps_its_sign_through_both_conversions(oracle_lib):
    """A NaN's sign comes from the input, not from the (platform-dependent) sign of
    a NaN product."""
    w = _conv_workload(40, num_layers=1, num_components=1, kv_heads=1, head_dim=16,
                       src_tp=1, dst_tp=1, src_block=4, dst_block=4, seq_lens=[2])
    src = [np.zeros(w.src_shape(), np.uint16)]
    rows = src[0].reshape(-1, 16)
    ids = w.src_bt[:1]
    v = src[0].reshape(w.src_num_blocks, 4, 16)
    v[ids[0], 0, :8] = 0x7FC1                        # +NaN
    v[ids[0], 0, 8:] = 0xFFC1                        # -NaN
    q = [np.zeros(w.dst_shape(), np.uint8)]
    oracle.relayout_convert(src, q, src_dtype=oracle.BF16, dst_dtype=oracle.E4M3, per_head=0,
                            scales=np.ones(1, np.float32), lib=oracle_lib, **_geometry(w))
    got = q[0].reshape(w.dst_num_blocks, 4, 16)[w.dst_bt[0], 0]
    assert list(got[:8]) == [0x7F] * 8 and list(got[8:]) == [0xFF] * 8
    w8 = dataclasses.replace(w, elem_bytes=1)
    codes = [np.zeros(w.src_shape(), np.uint8)]
    c = codes[0].reshape(w.src_num_blocks, 4, 16)
    c[ids[0], 0, :8] = 0x7F
    c[ids[0], 0, 8:] = 0xFF
    y = [np.zeros(w.dst_shape(), np.uint16)]
    oracle.relayout_convert(codes, y, src_dtype=oracle.E4M3, dst_dtype=oracle.BF16, per_head=0,
                            scales=np.ones(1, np.float32), lib=oracle_lib, **_geometry(w8))
    got = y[0].reshape(w.dst_num_blocks, 4, 16)[w.dst_bt[0], 0]
    assert list(got[:8]) == [0x7FC0] * 8 and list(got[8:]) == [0xFFC0] * 8
    del rows
