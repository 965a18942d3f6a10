"""Locate, build if needed, and load libpa.so; declare the C signatures."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

c_int, c_int64, c_size_t, c_float, c_void_p = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                               ctypes.c_float, ctypes.c_void_p)
P_I32 = ctypes.POINTER(ctypes.c_int32)
P_I64 = ctypes.POINTER(ctypes.c_int64)
P_INT = ctypes.POINTER(ctypes.c_int)


class PaBmStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "num_blocks", "free_blocks", "used_blocks", "shared_blocks", "num_seqs",
        "logical_blocks", "num_tokens", "waste_slots", "cow_copies")]


# name -> (restype, argtypes); mirrors include/pa.h
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [c_int]),
    "pa_abi_version": (c_int, []),
    "pa_reshape_and_cache": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                     c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pa_copy_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                               c_int, c_void_p]),
    "pa_decode_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "pa_decode_plan": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    "pa_decode": (c_int, [c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p,
                          c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                          c_float, c_void_p, c_size_t, c_void_p]),
    "pa_decode_append": (c_int, [c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_int, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                 c_int, c_float, c_void_p, c_size_t, c_void_p]),
    "pa_decode_shared_prefix_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int, c_int]),
    "pa_decode_shared_prefix": (c_int, [c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                        c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                        c_int, c_int, c_int, c_float, c_void_p, c_size_t, c_void_p]),
    "pa_decode_contiguous": (c_int, [c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                     c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                     c_void_p, c_size_t, c_void_p]),
    "pa_decode_static_scratch": (c_int, [c_void_p, c_int, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                         c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                         c_int, c_int, c_int, c_float, c_void_p]),
    "pa_decode_splitk": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p,
                                 c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_int, c_int, c_float, c_void_p]),
    "pa_lse_merge": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                             c_int, c_int, c_int, c_int, c_void_p]),
    "pa_device_status": (c_int, [P_INT, c_int, c_void_p]),
    "pa_check_wait_timeout": (c_int, [ctypes.c_uint, c_void_p]),
    "pa_compute_slot_mapping": (c_int, [P_I64, P_I32, c_int, c_int, P_I32, P_I32, c_int, c_int]),
    "pa_bm_create": (c_int, [c_int, c_int, c_int, ctypes.POINTER(c_void_p)]),
    "pa_bm_create_with_free_list": (c_int, [c_int, c_int, P_I32, c_int, ctypes.POINTER(c_void_p)]),
    "pa_bm_destroy": (None, [c_void_p]),
    "pa_bm_allocate": (c_int, [c_void_p, c_int64, c_int]),
    "pa_bm_append_slot": (c_int, [c_void_p, c_int64, P_I64, P_I64, P_I64]),
    "pa_bm_fork": (c_int, [c_void_p, c_int64, c_int64]),
    "pa_bm_free": (c_int, [c_void_p, c_int64]),
    "pa_bm_block_table": (c_int, [c_void_p, c_int64, P_I32, c_int, P_INT]),
    "pa_bm_num_tokens": (c_int, [c_void_p, c_int64, P_INT]),
    "pa_bm_refcount": (c_int, [c_void_p, c_int, P_INT]),
    "pa_bm_stats": (c_int, [c_void_p, ctypes.POINTER(PaBmStats)]),
    "pa_bm_free_list": (c_int, [c_void_p, P_I32, c_int, P_INT]),
    "pa_bm_enable_swap": (c_int, [c_void_p, c_int]),
    "pa_bm_swap_out": (c_int, [c_void_p, P_I64, c_int, P_I64, c_int, P_INT]),
    "pa_bm_swap_in": (c_int, [c_void_p, P_I64, c_int, P_I64, c_int, P_INT]),
    "pa_bm_is_swapped": (c_int, [c_void_p, c_int64, P_INT]),
    "pa_bm_swap_stats": (c_int, [c_void_p, P_I64, P_I64, P_I64]),
    "pa_swap_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                               c_int, c_int, c_int, c_void_p]),
}


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpa.so, building it first if it is missing or stale.

    Raises if the library cannot be built or loaded: there is no other
    implementation to fall back to."""
    global _lib
    lib = _lib
    if lib is not None:   # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libpa.so not found at {path}")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
