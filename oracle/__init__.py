"""CPU oracle for the prefill -> decode KV-cache relayout.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference legs of ``bench.py`` may import this package. The CUDA
library in ``prefill_decode_paged_gb300`` never imports it, and it imports
nothing from there.

Two independent definitions live here:

* ``kv_oracle.c`` (loaded through ctypes): the per-element loop nest over
  (request, layer, component, token, head, dim) that follows pd.py's
  ``prefill()`` gather and ``admit()`` slot formula on the page
  "PD 分离与 KV 传输" (section "实现"), with the TP head split of section
  "布局转换".
* ``pd_pages.py`` (numpy): the same hand-off written the way pd.py stages it,
  a gather of each layer into a contiguous ``[seq, kv_heads, head_dim]`` array
  followed by a write through a list of decode slots. It is only used on
  small inputs, as a cross-check of the C loop nest.

The converting relayout (``relayout_convert``: BF16 <-> FP8 E4M3 with a
scale, section "布局转换") and the layout-generic relayout
(``relayout_general``: any [block][token][head][dim] views per shard, layer
and component, same section) are further loop nests in ``kv_oracle.c``.

Parity status: every function is pinned against the pages and the
mathematics, not against itself: ``tests/test_oracle_pins.py`` (byte counts,
tagged brute force, inverse re-shard, reduction to a copy, the pd.py
restatement), ``tests/test_oracle_convert_pins.py`` (E4M3 decode at fixed points and
against torch's float8_e4m3fn, encode against torch, saturation and NaN,
BF16 rounding against torch, placement reduced to a copy of codes or values,
NaN signs through both directions), ``tests/test_oracle_layout_pins.py``
(standard views reduce to ``relayout`` and ``relayout_convert``; head-major
blocks, per-layer buffers, K/V interleaving and the staging buffer against
transposes and pd.py's gather) and
``tests/test_oracle_mutants.py`` (planted mistakes that the pins must catch).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkv_oracle.so")
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``kv_oracle.c`` with gcc into a shared library; return its path."""
    if not force and out == _LIB_PATH and os.path.exists(out) and (
            os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, src, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.kvo_bytes_per_token.restype = i64
    lib.kvo_bytes_per_token.argtypes = [i32, i32, i32, i32, i32]
    lib.kvo_transfer_bytes.restype = i64
    lib.kvo_transfer_bytes.argtypes = [i32, i32, i32, i32, i32, i32, p]
    lib.kvo_relayout.restype = ctypes.c_int
    lib.kvo_relayout.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                 i64, i64, p, p, i32, p, p, p, p, p]
    lib.kvo_relayout_general.restype = ctypes.c_int
    lib.kvo_relayout_general.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, p,
                                         i32, i32, i32, i32, p, i64, i64, i64, p, i64, i64,
                                         i64, i32, p, p, p, p, p]
    lib.kvo_relayout_convert.restype = ctypes.c_int
    lib.kvo_relayout_convert.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, p, i32,
                                         i32, i32, i32, i64, i64, p, p, i32, p, p, p, p, p]
    for name, t in (("kvo_e4m3_encode_array", None), ("kvo_e4m3_decode_array", None),
                    ("kvo_bf16_encode_array", None)):
        getattr(lib, name).restype = None
        getattr(lib, name).argtypes = [p, p, i64]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed).

    ``path`` loads another build of the same source (the mutation tests use
    this); the default build is cached.
    """
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def bytes_per_token(num_layers, num_components, kv_heads, head_dim, elem_bytes, lib=None):
    lib = lib or load()
    return int(lib.kvo_bytes_per_token(num_layers, num_components, kv_heads, head_dim,
                                       elem_bytes))


def transfer_bytes(num_layers, num_components, kv_heads, head_dim, elem_bytes, seq_lens,
                   lib=None):
    lib = lib or load()
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    return int(lib.kvo_transfer_bytes(num_layers, num_components, kv_heads, head_dim,
                                      elem_bytes, len(lens), lens.ctypes.data))


# dtype codes of the converting relayout
BF16 = 1
E4M3 = 2


def e4m3_encode(x, lib=None):
    """fp32 values -> E4M3 codes (nearest, ties to even, saturating at +-448)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib.kvo_e4m3_encode_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def e4m3_decode(codes, lib=None):
    lib = lib or load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float32)
    lib.kvo_e4m3_decode_array(c.ctypes.data, out.ctypes.data, c.size)
    return out


def bf16_encode(x, lib=None):
    """fp32 values -> bf16 bit patterns (nearest, ties to even)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.kvo_bf16_encode_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def _ptr_array(arrays, writable: bool):
    ptrs = (ctypes.c_void_p * max(1, len(arrays)))()
    for i, a in enumerate(arrays):
        if not a.flags.c_contiguous or (writable and not a.flags.writeable):
            raise ValueError("oracle pools must be C-contiguous (and writable on the dst side)")
        ptrs[i] = a.ctypes.data
    return ptrs


def relayout(src_pools, dst_pools, *, num_layers, num_components, kv_heads, head_dim,
             elem_bytes, src_tp, dst_tp, src_block, dst_block, src_num_blocks,
             dst_num_blocks, seq_lens, src_off, src_bt, dst_off, dst_bt,
             layer_begin=0, layer_end=None, lib=None):
    """Run the C oracle in place on numpy pools (one array per TP shard).

    ``src_off``/``dst_off`` are CSR offsets (int64, length R+1) into the flat
    block tables ``src_bt``/``dst_bt`` (int32). Layers [layer_begin,
    layer_end) are processed; the pools may also be single-layer slices, with
    ``num_layers=1`` and the layer range [0, 1).
    """
    lib = lib or load()
    if layer_end is None:
        layer_end = num_layers
    if len(src_pools) != src_tp or len(dst_pools) != dst_tp:
        raise ValueError("one pool per TP shard is required")
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    so = np.ascontiguousarray(src_off, dtype=np.int64)
    sb = np.ascontiguousarray(src_bt, dtype=np.int32)
    do = np.ascontiguousarray(dst_off, dtype=np.int64)
    db = np.ascontiguousarray(dst_bt, dtype=np.int32)
    # keep the (possibly empty) tables alive and non-null for the C side
    sb = sb if sb.size else np.zeros(1, np.int32)
    db = db if db.size else np.zeros(1, np.int32)
    sp = _ptr_array(src_pools, False)
    dp = _ptr_array(dst_pools, True)
    rc = lib.kvo_relayout(layer_begin, layer_end, num_layers, num_components, kv_heads,
                          head_dim, elem_bytes, src_tp, dst_tp, src_block, dst_block,
                          src_num_blocks, dst_num_blocks, sp, dp, len(lens),
                          lens.ctypes.data, so.ctypes.data, sb.ctypes.data, do.ctypes.data,
                          db.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the geometry (status {rc})")


def relayout_convert(src_pools, dst_pools, *, num_layers, num_components, kv_heads, head_dim,
                     src_dtype, dst_dtype, per_head, scales, src_tp, dst_tp, src_block,
                     dst_block, src_num_blocks, dst_num_blocks, seq_lens, src_off, src_bt,
                     dst_off, dst_bt, layer_begin=0, layer_end=None, lib=None, **_ignored):
    """The converting relayout (BF16 <-> E4M3) of the C oracle, in place on numpy pools."""
    lib = lib or load()
    if layer_end is None:
        layer_end = num_layers
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    so = np.ascontiguousarray(src_off, dtype=np.int64)
    sb = np.ascontiguousarray(src_bt, dtype=np.int32)
    do = np.ascontiguousarray(dst_off, dtype=np.int64)
    db = np.ascontiguousarray(dst_bt, dtype=np.int32)
    sb = sb if sb.size else np.zeros(1, np.int32)
    db = db if db.size else np.zeros(1, np.int32)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    sp = _ptr_array(src_pools, False)
    dp = _ptr_array(dst_pools, True)
    rc = lib.kvo_relayout_convert(layer_begin, layer_end, num_layers, num_components, kv_heads,
                                  head_dim, src_dtype, dst_dtype, int(per_head), sc.ctypes.data,
                                  src_tp, dst_tp, src_block, dst_block, src_num_blocks,
                                  dst_num_blocks, sp, dp, len(lens), lens.ctypes.data,
                                  so.ctypes.data, sb.ctypes.data, do.ctypes.data,
                                  db.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the conversion (status {rc})")


def _views_table(views, tp, num_layers, num_components):
    """Bases and shared (block, token, head) byte strides of [shard][layer][comp] views."""
    bases = np.zeros(tp * num_layers * num_components, dtype=np.uint64)
    strides = None
    for sh in range(tp):
        for l in range(num_layers):
            for c in range(num_components):
                v = views[sh][l][c]
                if v.ndim != 4 or v.strides[3] != v.itemsize:
                    raise ValueError("each view must be [block][token][head][dim], dim contiguous")
                if strides is None:
                    strides = v.strides[:3]
                elif v.strides[:3] != strides:
                    raise ValueError("all views of a side must share their strides")
                bases[(sh * num_layers + l) * num_components + c] = v.ctypes.data
    return bases, strides


def relayout_general(src_views, dst_views, *, num_layers, num_components, kv_heads, head_dim,
                     src_tp, dst_tp, src_block, dst_block, seq_lens, src_off, src_bt, dst_off,
                     dst_bt, elem_bytes=None, src_dtype=0, dst_dtype=0, per_head=0,
                     scales=None, layer_begin=0, layer_end=None, lib=None, **_ignored):
    """The oracle on any layout. ``src_views[s][l][c]`` / ``dst_views[s][l][c]`` are numpy
    views [block][token][head][dim] (dim contiguous) of the shard/layer/component's
    pool; they are written in place on the destination side."""
    lib = lib or load()
    if layer_end is None:
        layer_end = num_layers
    sb_, ss = _views_table(src_views, src_tp, num_layers, num_components)
    db_, ds = _views_table(dst_views, dst_tp, num_layers, num_components)
    if elem_bytes is None:
        elem_bytes = src_views[0][0][0].itemsize
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    so = np.ascontiguousarray(src_off, dtype=np.int64)
    sbt = np.ascontiguousarray(src_bt, dtype=np.int32)
    do = np.ascontiguousarray(dst_off, dtype=np.int64)
    dbt = np.ascontiguousarray(dst_bt, dtype=np.int32)
    sbt = sbt if sbt.size else np.zeros(1, np.int32)
    dbt = dbt if dbt.size else np.zeros(1, np.int32)
    sc = np.ascontiguousarray(scales if scales is not None else [1.0], dtype=np.float32)
    rc = lib.kvo_relayout_general(layer_begin, layer_end, num_layers, num_components, kv_heads,
                                  head_dim, src_dtype, dst_dtype, elem_bytes, int(per_head),
                                  sc.ctypes.data, src_tp, dst_tp, src_block, dst_block,
                                  sb_.ctypes.data, ss[0], ss[1], ss[2], db_.ctypes.data, ds[0],
                                  ds[1], ds[2], len(lens), lens.ctypes.data, so.ctypes.data,
                                  sbt.ctypes.data, do.ctypes.data, dbt.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the request (status {rc})")


def standard_views(pools, num_layers, num_components, num_blocks, block, heads, head_dim):
    """[shard][layer][comp] views of pools in the layout [L][C][N][B][H/T][D]."""
    out = []
    for p in pools:
        v = p.reshape(num_layers, num_components, num_blocks, block, heads, head_dim)
        out.append([[v[l, c] for c in range(num_components)] for l in range(num_layers)])
    return out
