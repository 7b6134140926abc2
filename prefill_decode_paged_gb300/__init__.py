"""GB300-native prefill -> decode KV-cache relayout (one fused sm_103a kernel behind a C ABI).

Public API (see ``include/kv_relayout.h`` for the C ABI it binds):

* :class:`RelayoutPlan` -- validate a batch and upload its work list;
  ``run_all()`` moves every layer in one launch, ``run_layer(l)`` one layer,
  ``run_layers(first, count)`` a range of layers; ``launch_shape`` reports the
  grids it chose.
* :func:`desc_bytes` -- host-only validation and byte count.
* :func:`layout_of_views` -- describe any physical layout (per-layer tensors, K/V
  interleaved, head-major blocks ...) for ``RelayoutPlan(src_layout=..., dst_layout=...)``.
* :func:`pack_plan` / :func:`unpack_plan` -- through a contiguous staging buffer
  ([L][C][tokens][H][D], pd.py's gathered shape).
* :class:`SmStream` -- a stream limited to a number of SMs (green context), to run
  the relayout beside other kernels.
* :func:`relayout_all_prealloc` -- ``run_all`` without any device allocation, for
  callers that cannot allocate (work lists up to 1 MiB).
* ``kv_relayout.checked_library()`` / ``build.build_checked()`` -- the same C ABI
  built with device-side address checks (tests).
"""
from .kv_relayout import (KVRelayoutError, RelayoutPlan, desc_bytes, library,  # noqa: F401
                          LIB_PATH, STATUS, EXPORTS, relayout_all_prealloc, layout_of_views,
                          pack_plan, unpack_plan, SmStream)
