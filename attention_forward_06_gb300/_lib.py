"""ctypes loading of the in-tree CUDA libraries (argument marshalling only).

The libraries are built by ``attention_forward_06_gb300.build`` into ``_build/``.
Loading fails loudly when a library is missing: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_libs: dict[str, ctypes.CDLL] = {}

_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p

# name -> (restype, argtypes), mirroring include/attn_fwd.h, include/attn_fwd_trace.h, include/attn_bwd.h,
# include/attn_bwd_trace.h and include/attn_fwd_probe.h
SIGNATURES = {
    "attn_fwd": {
        "attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _vp]),
        "attn_fwd_strerror": (ctypes.c_char_p, [_c_int]),
        "attn_fwd_version": (_c_int, []),
        "attn_fwd_debug_status": (_c_int, [_vp, ctypes.POINTER(_c_int)]),
        "attn_fwd_splitkv": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _c_int, _vp,
                                                                                  ctypes.c_size_t, _vp]),
        "attn_fwd_splitkv_workspace_size": (ctypes.c_size_t, [_c_int] * 5),
        "attn_fwd_splitkv_suggest": (_c_int, [_c_int] * 6),
        "attn_fwd_splitkv_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _c_int, _vp]),
        "attn_fwd_blocksparse": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _vp, _c_int, _vp]),
        "attn_fwd_block_mask_words": (ctypes.c_size_t, [_c_int] * 4),
        "attn_fwd_ordered": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _vp, _c_int, _vp]),
        "attn_fwd_tile_order_entries": (ctypes.c_size_t, [_c_int] * 4),
    },
    "attn_fwd_trace": {},  # filled below: attn_fwd's entry points and the trace reader
    "attn_bwd": {
        "attn_bwd": (_c_int, [_vp] * 9 + [_c_int] * 7 + [_c_float, _vp, ctypes.c_size_t, _vp]),
        "attn_bwd_workspace_size": (ctypes.c_size_t, [_c_int] * 3),
        "attn_bwd_strerror": (ctypes.c_char_p, [_c_int]),
        "attn_bwd_debug_status": (_c_int, [_vp, ctypes.POINTER(_c_int)]),
    },
    "attn_probe": {
        "attn_probe_mma_ss": (_c_int, [_vp, _c_int, _vp, _c_int, _c_int, _vp, _vp, _vp, _vp]),
        "attn_probe_mma_ts": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
        "attn_probe_wait_timeout": (_c_int, [ctypes.c_ulonglong, ctypes.c_ulonglong, _vp, _vp, _vp]),
        "attn_probe_mma_rate": (_c_int, [_c_int, _c_int, _c_int, _vp, _vp, _vp, _vp]),
        "attn_probe_ex2_rate": (_c_int, [_c_int, _c_int, _vp, _vp, _vp]),
    },
}


SIGNATURES["attn_fwd_trace"] = dict(SIGNATURES["attn_fwd"])
SIGNATURES["attn_fwd_trace"]["attn_fwd_trace_read"] = (
    _c_int, [_vp, ctypes.c_size_t, ctypes.POINTER(_c_int), ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)])
SIGNATURES["attn_bwd_trace"] = dict(SIGNATURES["attn_bwd"])
SIGNATURES["attn_bwd_trace"]["attn_bwd_trace_read"] = (
    _c_int, [_vp, ctypes.c_size_t] + [ctypes.POINTER(_c_int)] * 4)


class LibraryMissing(RuntimeError):
    pass


def load(name: str = "attn_fwd", build_if_missing: bool = False) -> ctypes.CDLL:
    """Load ``lib<name>.so`` from ``_build/`` and set its function signatures."""
    with _lock:
        if name in _libs:
            return _libs[name]
        path = _build.lib_path(name)
        if not os.path.exists(path):
            if not build_if_missing:
                raise LibraryMissing(
                    f"{path} is missing: build it with `python -m attention_forward_06_gb300.build` "
                    "(the CUDA path has no fallback)")
            _build.build()
        lib = ctypes.CDLL(path)
        for fn, (res, args) in SIGNATURES[name].items():
            f = getattr(lib, fn)
            f.restype = res
            f.argtypes = args
        _libs[name] = lib
        return lib
