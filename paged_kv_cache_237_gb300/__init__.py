"""GB300-native paged decode attention (PagedAttention hot path).

The compute path is a C-ABI shared library (``csrc/``, declared in
``include/pa.h``) of hand-written sm_103a CUDA kernels:

- ``pa_decode``: decode-step attention over a KV cache held in fixed-size
  physical blocks reached through a per-sequence block table, with a split-K
  reduce for long contexts;
- ``pa_reshape_and_cache``: writes each new token's K/V into its physical slot;
- ``pa_copy_blocks``: whole-block copies behind copy-on-write;
- ``pa_swap_blocks``: whole-block copies between a device pool and pinned host memory;

plus a host block manager (free pool, refcounts, copy-on-write trigger, prefix cache, moves between pools).

``binding`` is the thin ctypes layer with the same names.  It is imported
lazily so that ``workloads`` can be used without the compiled library; any use
of a compute entry point without the library raises ``ImportError``.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = {
    "pa_decode", "pa_decode_workspace_size", "pa_reshape_and_cache", "pa_copy_blocks", "pa_swap_blocks",
    "BlockManager", "DeviceStatus", "PAError", "library_path", "load_library",
    "PA_PHASE_ALL", "PA_PHASE_PARTITIONS", "PA_PHASE_REDUCE",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
