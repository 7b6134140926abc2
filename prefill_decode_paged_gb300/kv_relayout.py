"""ctypes binding of the C ABI in ``include/kv_relayout.h`` (argument marshalling only).

Every step of the relayout runs in the CUDA library ``_build/libkv_relayout.so``;
this module only converts Python/numpy/torch arguments into the C descriptor
and forwards the calls. There is no fallback: if the library is missing or a
call fails, it raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libkv_relayout.so")
MAX_TP = 16

STATUS = {
    0: "KVR_OK", -1: "KVR_ERR_INVALID_ARG", -2: "KVR_ERR_UNSUPPORTED",
    -3: "KVR_ERR_ALIGNMENT", -4: "KVR_ERR_BLOCK_RANGE", -5: "KVR_ERR_TABLE_SHORT",
    -6: "KVR_ERR_DST_ALIAS", -7: "KVR_ERR_LAYER_RANGE", -8: "KVR_ERR_CUDA",
    -9: "KVR_ERR_NOMEM", -10: "KVR_ERR_POOL_OVERLAP", -11: "KVR_ERR_SCRATCH_LIMIT",
    -12: "KVR_ERR_POOL_ADDRESS",
}
PREALLOC_SCRATCH_BYTES = 1 << 20
EXPORTS = ("kv_relayout_desc_bytes", "kv_relayout_plan", "kv_relayout_layer",
           "kv_relayout_all", "kv_relayout_plan_bytes", "kv_relayout_plan_destroy",
           "kv_relayout_strerror", "kv_relayout_all_prealloc", "kv_relayout_desc_convert_bytes",
           "kv_relayout_plan_convert")
DTYPE_BF16 = 1
DTYPE_FP8_E4M3 = 2


class KVRelayoutError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.name} ({_strerror(status)})")


class KvrConvert(ctypes.Structure):
    _fields_ = [("src_dtype", ctypes.c_int32), ("dst_dtype", ctypes.c_int32),
                ("per_head", ctypes.c_int32), ("scales", ctypes.c_void_p)]


class KvrDesc(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_components", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("elem_bytes", ctypes.c_int32), ("src_tp", ctypes.c_int32),
        ("dst_tp", ctypes.c_int32), ("src_block_size", ctypes.c_int32),
        ("dst_block_size", ctypes.c_int32), ("src_num_blocks", ctypes.c_int64),
        ("dst_num_blocks", ctypes.c_int64), ("src_pools", ctypes.c_void_p),
        ("dst_pools", ctypes.c_void_p), ("num_requests", ctypes.c_int32),
        ("seq_lens", ctypes.c_void_p), ("src_bt_offsets", ctypes.c_void_p),
        ("src_bt", ctypes.c_void_p), ("dst_bt_offsets", ctypes.c_void_p),
        ("dst_bt", ctypes.c_void_p),
    ]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library {LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        lib.kv_relayout_desc_bytes.restype = i32
        lib.kv_relayout_desc_bytes.argtypes = [p, p, p]
        lib.kv_relayout_plan.restype = i32
        lib.kv_relayout_plan.argtypes = [p, p]
        lib.kv_relayout_layer.restype = i32
        lib.kv_relayout_layer.argtypes = [p, i32, p]
        lib.kv_relayout_all.restype = i32
        lib.kv_relayout_all.argtypes = [p, p]
        lib.kv_relayout_plan_bytes.restype = i32
        lib.kv_relayout_plan_bytes.argtypes = [p, p, p]
        lib.kv_relayout_plan_destroy.restype = None
        lib.kv_relayout_plan_destroy.argtypes = [p]
        lib.kv_relayout_strerror.restype = ctypes.c_char_p
        lib.kv_relayout_strerror.argtypes = [i32]
        lib.kv_relayout_all_prealloc.restype = i32
        lib.kv_relayout_all_prealloc.argtypes = [p, p]
        lib.kv_relayout_desc_convert_bytes.restype = i32
        lib.kv_relayout_desc_convert_bytes.argtypes = [p, p, p, p]
        lib.kv_relayout_plan_convert.restype = i32
        lib.kv_relayout_plan_convert.argtypes = [p, p, p]
        _lib = lib
    return _lib


def _strerror(status: int) -> str:
    try:
        return library().kv_relayout_strerror(status).decode()
    except Exception:  # the message is best effort; the status is what matters
        return "?"


def _ptr(x) -> int:
    """Device address of a torch tensor (or an int that already is one)."""
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


class _Desc:
    """Keeps the C descriptor and every host array it points to alive."""

    def __init__(self, src_pools, dst_pools, *, num_layers, num_components, kv_heads,
                 head_dim, elem_bytes, src_tp, dst_tp, src_block, dst_block, src_num_blocks,
                 dst_num_blocks, seq_lens, src_off, src_bt, dst_off, dst_bt):
        if src_pools is not None and len(src_pools) > MAX_TP or \
                dst_pools is not None and len(dst_pools) > MAX_TP:
            raise ValueError(f"at most {MAX_TP} shard pools per side")
        self.src = (ctypes.c_void_p * MAX_TP)(*[_ptr(x) for x in (src_pools or [])])
        self.dst = (ctypes.c_void_p * MAX_TP)(*[_ptr(x) for x in (dst_pools or [])])
        self.lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        self.soff = np.ascontiguousarray(src_off, dtype=np.int64)
        self.sbt = np.ascontiguousarray(src_bt, dtype=np.int32)
        self.doff = np.ascontiguousarray(dst_off, dtype=np.int64)
        self.dbt = np.ascontiguousarray(dst_bt, dtype=np.int32)
        d = KvrDesc()
        d.num_layers, d.num_components, d.kv_heads = num_layers, num_components, kv_heads
        d.head_dim, d.elem_bytes = head_dim, elem_bytes
        d.src_tp, d.dst_tp = src_tp, dst_tp
        d.src_block_size, d.dst_block_size = src_block, dst_block
        d.src_num_blocks, d.dst_num_blocks = src_num_blocks, dst_num_blocks
        d.src_pools = ctypes.cast(self.src, ctypes.c_void_p) if src_pools is not None else None
        d.dst_pools = ctypes.cast(self.dst, ctypes.c_void_p) if dst_pools is not None else None
        d.num_requests = len(self.lens)
        d.seq_lens = self.lens.ctypes.data if self.lens.size else None
        d.src_bt_offsets = self.soff.ctypes.data if self.soff.size else None
        d.src_bt = self.sbt.ctypes.data if self.sbt.size else None
        d.dst_bt_offsets = self.doff.ctypes.data if self.doff.size else None
        d.dst_bt = self.dbt.ctypes.data if self.dbt.size else None
        self.desc = d


class _Convert:
    """Keeps the C conversion descriptor and its scales alive."""

    def __init__(self, src_dtype, dst_dtype, scales, per_head=False):
        self.scales = np.ascontiguousarray(scales, dtype=np.float32)
        c = KvrConvert()
        c.src_dtype, c.dst_dtype, c.per_head = int(src_dtype), int(dst_dtype), int(per_head)
        c.scales = self.scales.ctypes.data if self.scales.size else None
        self.conv = c


def desc_bytes(src_pools, dst_pools, convert=None, **geometry):
    """Validate a descriptor on the host; return (bytes_read, bytes_written)."""
    d = _Desc(src_pools, dst_pools, **geometry)
    r, w = ctypes.c_int64(), ctypes.c_int64()
    if convert is None:
        st = library().kv_relayout_desc_bytes(ctypes.byref(d.desc), ctypes.byref(r),
                                              ctypes.byref(w))
    else:
        cv = _Convert(**convert)
        st = library().kv_relayout_desc_convert_bytes(ctypes.byref(d.desc),
                                                      ctypes.byref(cv.conv), ctypes.byref(r),
                                                      ctypes.byref(w))
    if st != 0:
        raise KVRelayoutError(st, "kv_relayout_desc_bytes")
    return r.value, w.value


def relayout_all_prealloc(src_pools, dst_pools, stream=None, **geometry):
    """All layers in one launch without any device allocation.

    For callers that cannot call cudaMalloc while handing KV over (an engine
    whose HBM is already carved into KV pools, a loop that cannot afford the
    device-wide synchronization of cudaMalloc/cudaFree). The work list goes
    into a fixed 1 MiB device array the library keeps on every GPU it runs on;
    larger work lists raise ``KVR_ERR_SCRATCH_LIMIT`` (use :class:`RelayoutPlan`).
    The first call on a device sets the array up and should come before any
    stream capture. Calls share the array: calls that overlap on the GPU (on
    different, unordered streams) race.
    """
    d = _Desc(src_pools, dst_pools, **geometry)
    st = library().kv_relayout_all_prealloc(ctypes.byref(d.desc), _stream_handle(stream))
    if st != 0:
        raise KVRelayoutError(st, "kv_relayout_all_prealloc")


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


class RelayoutPlan:
    """A validated relayout of one batch of prompts, ready to launch.

    ``src_pools``/``dst_pools``: one device buffer (torch tensor or address)
    per TP shard, layout [L][C][N][B][H / tp][D]. Block tables are CSR:
    ``src_off``/``dst_off`` (R + 1 offsets) into ``src_bt``/``dst_bt``.
    ``convert``: None (bit copy) or dict(src_dtype=..., dst_dtype=..., scales=...,
    per_head=False) for a BF16 <-> FP8 E4M3 relayout (``kv_relayout_plan_convert``).
    """

    def __init__(self, src_pools, dst_pools, convert=None, **geometry):
        self._h = None
        self._d = _Desc(src_pools, dst_pools, **geometry)
        self.num_layers = geometry["num_layers"]
        h = ctypes.c_void_p()
        if convert is None:
            st = library().kv_relayout_plan(ctypes.byref(self._d.desc), ctypes.byref(h))
        else:
            self._cv = _Convert(**convert)
            st = library().kv_relayout_plan_convert(ctypes.byref(self._d.desc),
                                                    ctypes.byref(self._cv.conv), ctypes.byref(h))
        if st != 0:
            raise KVRelayoutError(st, "kv_relayout_plan")
        self._h = h
        r, w = ctypes.c_int64(), ctypes.c_int64()
        st = library().kv_relayout_plan_bytes(self._h, ctypes.byref(r), ctypes.byref(w))
        if st != 0:
            raise KVRelayoutError(st, "kv_relayout_plan_bytes")
        self.bytes_read, self.bytes_written = r.value, w.value

    def run_all(self, stream=None):
        """All layers, one launch on ``stream`` (default: torch's current stream)."""
        st = library().kv_relayout_all(self._handle(), _stream_handle(stream))
        if st != 0:
            raise KVRelayoutError(st, "kv_relayout_all")

    def run_layer(self, layer: int, stream=None):
        """One layer, one launch on ``stream`` (default: torch's current stream)."""
        st = library().kv_relayout_layer(self._handle(), int(layer), _stream_handle(stream))
        if st != 0:
            raise KVRelayoutError(st, "kv_relayout_layer")

    def _handle(self):
        if self._h is None:
            raise RuntimeError("plan already closed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None:
            library().kv_relayout_plan_destroy(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
