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
    -12: "KVR_ERR_POOL_ADDRESS", -13: "KVR_ERR_DEVICE_BOUNDS",
}
PREALLOC_SCRATCH_BYTES = 1 << 20
EXPORTS = ("kv_relayout_desc_bytes", "kv_relayout_plan", "kv_relayout_layer",
           "kv_relayout_all", "kv_relayout_plan_bytes", "kv_relayout_plan_destroy",
           "kv_relayout_strerror", "kv_relayout_all_prealloc", "kv_relayout_desc_convert_bytes",
           "kv_relayout_plan_convert", "kv_relayout_desc_bytes_ex", "kv_relayout_plan_ex",
           "kv_relayout_sm_stream_create", "kv_relayout_sm_stream_destroy",
           "kv_relayout_plan_launch_shape", "kv_relayout_layers", "kv_relayout_layers_ex",
           "kv_relayout_debug_status", "kv_relayout_debug_narrow",
           "kv_relayout_staging_bytes", "kv_relayout_plan_pack", "kv_relayout_plan_unpack")
DTYPE_BF16 = 1
DTYPE_FP8_E4M3 = 2
LAUNCH_NO_WAIT = 1


class KVRelayoutError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.name} ({_strerror(status)})")


class KvrConvert(ctypes.Structure):
    _fields_ = [("src_dtype", ctypes.c_int32), ("dst_dtype", ctypes.c_int32),
                ("per_head", ctypes.c_int32), ("scales", ctypes.c_void_p)]


class KvrLayout(ctypes.Structure):
    _fields_ = [("bases", ctypes.c_void_p), ("block_stride", ctypes.c_int64),
                ("token_stride", ctypes.c_int64), ("head_stride", ctypes.c_int64)]


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
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def checked_library() -> ctypes.CDLL:
    """The library built with device-side address checks (tests only): the same C ABI,
    plus working ``kv_relayout_debug_status`` / ``kv_relayout_debug_narrow``. Builds it
    on first use. Call its functions directly with a ``_Desc``; ``RelayoutPlan`` uses
    the product library."""
    from . import build as kbuild
    return _bind(ctypes.CDLL(kbuild.build_checked()))


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures on a loaded copy of the library."""
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
    lib.kv_relayout_desc_bytes_ex.restype = i32
    lib.kv_relayout_desc_bytes_ex.argtypes = [p, p, p, p, p, p]
    lib.kv_relayout_plan_ex.restype = i32
    lib.kv_relayout_plan_ex.argtypes = [p, p, p, p, p]
    lib.kv_relayout_sm_stream_create.restype = i32
    lib.kv_relayout_sm_stream_create.argtypes = [i32, p, p, p]
    lib.kv_relayout_sm_stream_destroy.restype = None
    lib.kv_relayout_sm_stream_destroy.argtypes = [p]
    lib.kv_relayout_plan_launch_shape.restype = i32
    lib.kv_relayout_plan_launch_shape.argtypes = [p, p, p, p]
    lib.kv_relayout_layers.restype = i32
    lib.kv_relayout_layers.argtypes = [p, i32, i32, p]
    lib.kv_relayout_layers_ex.restype = i32
    lib.kv_relayout_layers_ex.argtypes = [p, i32, i32, ctypes.c_uint32, p]
    lib.kv_relayout_debug_status.restype = i32
    lib.kv_relayout_debug_status.argtypes = [p, p]
    lib.kv_relayout_debug_narrow.restype = i32
    lib.kv_relayout_debug_narrow.argtypes = [p, i64]
    lib.kv_relayout_staging_bytes.restype = i32
    lib.kv_relayout_staging_bytes.argtypes = [p, i32, p]
    lib.kv_relayout_plan_pack.restype = i32
    lib.kv_relayout_plan_pack.argtypes = [p, p, p, p]
    lib.kv_relayout_plan_unpack.restype = i32
    lib.kv_relayout_plan_unpack.argtypes = [p, p, p, p]
    return lib


def _strerror(status: int) -> str:
    try:
        return library().kv_relayout_strerror(status).decode()
    except Exception:  # the message is best effort; the status is what matters
        return "?"


def _ptr(x) -> int:
    """Address of a torch tensor or numpy array (or an int that already is one)."""
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x.ctypes.data)


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


class _Layout:
    """Keeps a C layout descriptor and its base-address array alive."""

    def __init__(self, bases, block_stride, token_stride, head_stride, shape=None,
                 elem_bytes=None):
        self.bases = (ctypes.c_void_p * max(1, len(bases)))(*[_ptr(x) for x in bases])
        lay = KvrLayout()
        lay.bases = ctypes.cast(self.bases, ctypes.c_void_p)
        lay.block_stride, lay.token_stride, lay.head_stride = (int(block_stride),
                                                              int(token_stride),
                                                              int(head_stride))
        self.layout = lay


def layout_of_views(views):
    """A side's layout from its views: ``views[shard][layer][component]`` are tensors
    (torch or numpy) shaped [block][token][head][dim] with a contiguous last
    dimension, the same strides and the same element size. Returns the dict
    RelayoutPlan takes; besides the bases and strides it records the views'
    smallest extents (``shape``) and element size, which the plan checks against
    the geometry (the C library sees addresses only)."""
    bases, strides, shape, elem = [], None, None, None
    for per_shard in views:
        for per_layer in per_shard:
            for v in per_layer:
                if hasattr(v, "data_ptr"):                       # torch
                    es = v.element_size()
                    st = tuple(x * es for x in v.stride())
                    bases.append(int(v.data_ptr()))
                else:                                            # numpy
                    es = v.itemsize
                    st = tuple(v.strides)
                    bases.append(int(v.ctypes.data))
                if len(st) != 4 or st[3] != es:
                    raise ValueError("views must be [block][token][head][dim], dim contiguous")
                if strides is None:
                    strides, shape, elem = st[:3], tuple(int(x) for x in v.shape), es
                elif st[:3] != strides or es != elem:
                    raise ValueError("all views of a side must share their strides and "
                                     "element size")
                else:
                    shape = tuple(min(a, int(b)) for a, b in zip(shape, v.shape))
    if strides is None:
        raise ValueError("no views")
    return dict(bases=bases, block_stride=strides[0], token_stride=strides[1],
                head_stride=strides[2], shape=shape, elem_bytes=elem)


_DTYPE_BYTES = {DTYPE_BF16: 2, DTYPE_FP8_E4M3: 1}


def _nbytes(x):
    """Bytes of a torch tensor or numpy array; None for a bare address."""
    if isinstance(x, int):
        return None
    if hasattr(x, "element_size") and hasattr(x, "numel"):
        return int(x.numel()) * int(x.element_size())
    if hasattr(x, "nbytes"):
        return int(x.nbytes)
    return None


def _contiguous(x) -> bool:
    if hasattr(x, "is_contiguous"):
        return bool(x.is_contiguous())
    flags = getattr(x, "flags", None)
    return flags is None or bool(flags["C_CONTIGUOUS"])


def _check_extents(src_pools, dst_pools, convert, src_layout, dst_layout, g):
    """The C library checks pool addresses, not allocation sizes: make sure every
    pool tensor and every described view holds what the geometry addresses, so an
    undersized tensor raises here instead of being written past its end. Geometry
    the library itself refuses (zero sizes, a TP degree that neither divides nor is a
    multiple of the head count) is left to it."""
    es_src = g["elem_bytes"]
    es_dst = es_src if convert is None else _DTYPE_BYTES.get(int(convert["dst_dtype"]), es_src)
    for side, pools, layout, es in (("src", src_pools, src_layout, es_src),
                                    ("dst", dst_pools, dst_layout, es_dst)):
        T, H = g[f"{side}_tp"], g["kv_heads"]
        if T < 1 or H < 1 or (H % T and T % H):
            continue
        # heads per shard: H / T, or 1 when T > H (each head held by T / H shards)
        need_shape = (g[f"{side}_num_blocks"], g[f"{side}_block"], max(H // T, 1),
                      g["head_dim"])
        if layout is not None:
            shape, elem = layout.get("shape"), layout.get("elem_bytes")
            if elem is not None and elem != es:
                raise ValueError(f"{side} views hold {elem}-byte elements; the relayout "
                                 f"{'reads' if side == 'src' else 'writes'} {es}-byte ones")
            if shape is not None and any(h < n for h, n in zip(shape, need_shape)):
                raise ValueError(f"{side} views are {list(shape)} ([block][token][head][dim]); "
                                 f"the geometry addresses {list(need_shape)}")
            continue
        if pools is None:
            continue
        need = g["num_layers"] * g["num_components"] * es
        for x in need_shape:
            need *= x
        for k, p in enumerate(pools):
            if not _contiguous(p):
                raise ValueError(f"{side} pool {k} is not contiguous: describe a strided "
                                 f"pool with a layout (layout_of_views)")
            have = _nbytes(p)
            if have is not None and have < need:
                raise ValueError(f"{side} pool {k} holds {have} bytes; the geometry "
                                 f"addresses {need}")


def _layout_arg(layout):
    return None if layout is None else _Layout(**layout)


def desc_bytes(src_pools, dst_pools, convert=None, src_layout=None, dst_layout=None,
               **geometry):
    """Validate a descriptor on the host; return (bytes_read, bytes_written)."""
    _check_extents(src_pools, dst_pools, convert, src_layout, dst_layout, geometry)
    d = _Desc(src_pools, dst_pools, **geometry)
    r, w = ctypes.c_int64(), ctypes.c_int64()
    if src_layout is not None or dst_layout is not None:
        sl, dl = _layout_arg(src_layout), _layout_arg(dst_layout)
        cv = _Convert(**convert) if convert is not None else None
        st = library().kv_relayout_desc_bytes_ex(
            ctypes.byref(d.desc), ctypes.byref(sl.layout) if sl else None,
            ctypes.byref(dl.layout) if dl else None, ctypes.byref(cv.conv) if cv else None,
            ctypes.byref(r), ctypes.byref(w))
    elif convert is None:
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
    stream capture; on a stream under capture the call raises
    ``KVR_ERR_UNSUPPORTED`` and enqueues nothing. Calls share the array: calls from
    several threads on one stream run one after another, calls that overlap on the
    GPU (on different, unordered streams) race.
    """
    _check_extents(src_pools, dst_pools, None, None, None, geometry)
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
    per TP shard, layout [L][C][N][B][H / tp][D] (a TP degree above H, a multiple
    of it: [L][C][N][B][1][D], tp / H shards per head). Block tables are CSR:
    ``src_off``/``dst_off`` (R + 1 offsets) into ``src_bt``/``dst_bt``.
    ``convert``: None (bit copy) or dict(src_dtype=..., dst_dtype=..., scales=...,
    per_head=False) for a BF16 <-> FP8 E4M3 relayout (``kv_relayout_plan_convert``).
    ``src_layout`` / ``dst_layout``: None (the pools in the standard layout) or a
    dict(bases=..., block_stride=..., token_stride=..., head_stride=...) as
    :func:`layout_of_views` builds (``kv_relayout_plan_ex``); the side's pools are
    then not used and may be None.
    """

    def __init__(self, src_pools, dst_pools, convert=None, src_layout=None, dst_layout=None,
                 **geometry):
        self._h = None
        _check_extents(src_pools, dst_pools, convert, src_layout, dst_layout, geometry)
        self._d = _Desc(src_pools, dst_pools, **geometry)
        self.num_layers = geometry["num_layers"]
        h = ctypes.c_void_p()
        if src_layout is not None or dst_layout is not None:
            self._sl, self._dl = _layout_arg(src_layout), _layout_arg(dst_layout)
            self._cv = _Convert(**convert) if convert is not None else None
            st = library().kv_relayout_plan_ex(
                ctypes.byref(self._d.desc),
                ctypes.byref(self._sl.layout) if self._sl else None,
                ctypes.byref(self._dl.layout) if self._dl else None,
                ctypes.byref(self._cv.conv) if self._cv else None, ctypes.byref(h))
        elif convert is None:
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

    @classmethod
    def _adopt(cls, handle, num_layers, keep):
        """Wrap a plan the library already made (``keep``: the host objects its
        descriptor pointed to, held for the plan's lifetime)."""
        self = cls.__new__(cls)
        self._h, self._keep, self.num_layers = handle, keep, num_layers
        r, w = ctypes.c_int64(), ctypes.c_int64()
        st = library().kv_relayout_plan_bytes(self._h, ctypes.byref(r), ctypes.byref(w))
        if st != 0:
            self.close()
            raise KVRelayoutError(st, "kv_relayout_plan_bytes")
        self.bytes_read, self.bytes_written = r.value, w.value
        return self

    @property
    def launch_shape(self):
        """(CTAs of one run_all launch, CTAs of one run_layer launch, tokens per tile)."""
        ga, gl, t = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        st = library().kv_relayout_plan_launch_shape(self._handle(), ctypes.byref(ga),
                                                     ctypes.byref(gl), ctypes.byref(t))
        if st != 0:
            raise KVRelayoutError(st, "kv_relayout_plan_launch_shape")
        return ga.value, gl.value, t.value

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

    def run_layers(self, first: int, count: int, stream=None, wait_for_previous=True):
        """Layers [first, first + count), one launch on ``stream`` (default: torch's
        current stream). ``wait_for_previous=False`` passes KVR_LAUNCH_NO_WAIT: only
        when the work just before this launch on the stream is another hand-off launch
        and everything this launch reads and writes was written by work queued before
        the latest hand-off launch made with ``wait_for_previous=True`` (see
        ``kv_relayout_layers_ex`` in the C header)."""
        flags = 0 if wait_for_previous else LAUNCH_NO_WAIT
        st = library().kv_relayout_layers_ex(self._handle(), int(first), int(count), flags,
                                             _stream_handle(stream))
        if st != 0:
            raise KVRelayoutError(st, "kv_relayout_layers")

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


class SmStream:
    """A stream whose kernels run on at most ~``sm_count`` SMs (a green context).

    ``handle`` is the cudaStream_t (an int) to pass as ``stream=`` to
    :meth:`RelayoutPlan.run_all` / :meth:`RelayoutPlan.run_layer`; wrap it with
    ``torch.cuda.ExternalStream(handle)`` to order it with torch work.
    ``sms`` is the number of SMs granted (rounded up to the split granularity).
    """

    def __init__(self, sm_count: int):
        self._h = ctypes.c_void_p()
        s, g = ctypes.c_void_p(), ctypes.c_int32()
        st = library().kv_relayout_sm_stream_create(int(sm_count), ctypes.byref(self._h),
                                                    ctypes.byref(s), ctypes.byref(g))
        if st != 0:
            self._h = None
            raise KVRelayoutError(st, "kv_relayout_sm_stream_create")
        self.handle, self.sms = s.value, g.value

    def close(self):
        if getattr(self, "_h", None) is not None:
            library().kv_relayout_sm_stream_destroy(self._h)
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


# -- staging buffer: pd.py's gathered [seq, kv_heads, head_dim] per layer ---------------

def staging_bytes(staging_elem_bytes, **geometry):
    """Bytes of the staging buffer [L][C][sum n][H][D] of ``staging_elem_bytes``-byte
    elements for this batch (``kv_relayout_staging_bytes``)."""
    d = _Desc(None, None, **geometry)
    out = ctypes.c_int64()
    st = library().kv_relayout_staging_bytes(ctypes.byref(d.desc), int(staging_elem_bytes),
                                             ctypes.byref(out))
    if st != 0:
        raise KVRelayoutError(st, "kv_relayout_staging_bytes")
    return out.value


def _check_staging(buf, convert, pack, geometry):
    """The staging tensor must be [L][C][sum n][H][D], contiguous, of the staging dtype."""
    L, C = geometry["num_layers"], geometry["num_components"]
    total = int(np.asarray(geometry["seq_lens"], dtype=np.int64).sum())
    want = (L, C, total, geometry["kv_heads"], geometry["head_dim"])
    if tuple(int(x) for x in buf.shape) != want:
        raise ValueError(f"staging buffer is {list(buf.shape)}; expected "
                         f"[{L}][{C}][{total}][heads][head_dim] = {list(want)}")
    if not _contiguous(buf):
        raise ValueError("staging buffer must be contiguous")
    es = geometry["elem_bytes"]
    if pack and convert is not None:
        es = _DTYPE_BYTES.get(int(convert["dst_dtype"]), es)
    have = _nbytes(buf)
    if have is not None and have != staging_bytes(es, **geometry):
        raise ValueError(f"staging buffer holds {have} bytes of "
                         f"{have // max(1, int(np.prod(want)))}-byte elements; the staging "
                         f"side holds {es}-byte elements")


def _staging_plan(pools, staging, convert, pack, geometry):
    if pack:
        _check_extents(pools, None, convert, None, {}, geometry)
    else:
        _check_extents(None, pools, convert, {}, None, geometry)
    _check_staging(staging, convert, pack, geometry)
    d = _Desc(pools if pack else None, None if pack else pools, **geometry)
    cv = _Convert(**convert) if convert is not None else None
    h = ctypes.c_void_p()
    fn = library().kv_relayout_plan_pack if pack else library().kv_relayout_plan_unpack
    st = fn(ctypes.byref(d.desc), _ptr(staging), ctypes.byref(cv.conv) if cv else None,
            ctypes.byref(h))
    if st != 0:
        raise KVRelayoutError(st, "kv_relayout_plan_pack" if pack else "kv_relayout_plan_unpack")
    return RelayoutPlan._adopt(h, geometry["num_layers"], keep=(d, cv, staging, pools))


def pack_plan(src_pools, staging, convert=None, **geometry):
    """Plan that gathers every request's KV out of the prefill pools into ``staging``
    ([L][C][sum n][H][D]: pd.py's per-layer [seq, kv_heads, head_dim], requests one
    after another), merging the prefill TP shards' heads (``kv_relayout_plan_pack``;
    the geometry's decode-side entries are not used)."""
    return _staging_plan(src_pools, staging, convert, True, geometry)


def unpack_plan(staging, dst_pools, convert=None, **geometry):
    """Plan that writes a staging buffer filled by :func:`pack_plan` into the decode
    pools through the decode block table, splitting heads over the decode TP shards
    (``kv_relayout_plan_unpack``; the geometry's prefill-side entries are not used)."""
    return _staging_plan(dst_pools, staging, convert, False, geometry)
