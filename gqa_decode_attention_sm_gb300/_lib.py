"""ctypes loader for libgqa_decode.so (argument types of the C ABI only).

There is no fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

_lib = None
_lock = threading.Lock()

# Every extern "C" function declared in include/gqa_decode.h.
EXPORTS = (
    "gqa_status_string", "gqa_last_error", "gqa_decode_workspace_size", "gqa_decode_plan",
    "gqa_decode_plan_for", "gqa_decode_split_geometry", "gqa_decode_launch_count_for",
    "gqa_decode", "gqa_decode_prepared", "gqa_decode_fp8kv", "gqa_decode_split_stage",
    "gqa_decode_combine_stage", "gqa_decode_workspace_init", "gqa_decode_get_status",
    "gqa_decode_noalloc", "gqa_decode_noalloc_get_status", "gqa_decode_debug_skip_tile",
    "gqa_decode_debug_cut_extents", "gqa_decode_int8kv", "gqa_decode_paged",
    "gqa_decode_verify", "gqa_append_kv", "gqa_append_kv_paged",
)


class GqaError(RuntimeError):
    def __init__(self, status: int, name: str, message: str):
        super().__init__(f"{name}: {message}" if message else name)
        self.status = status
        self.name = name


def _declare(lib):
    p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "gqa_status_string": (ctypes.c_char_p, [i]),
        "gqa_last_error": (ctypes.c_char_p, []),
        "gqa_decode_workspace_size": (sz, [i, i, i]),
        "gqa_decode_plan": (i, [i, i, i, i, ctypes.POINTER(ctypes.c_int)]),
        "gqa_decode_plan_for": (i, [i, i, i, i, ctypes.POINTER(ctypes.c_int)]),
        "gqa_decode_split_geometry": (i, [i, i, i, ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(ctypes.c_int)]),
        "gqa_decode_launch_count_for": (i, [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]),
        "gqa_decode": (i, [p, p, p, p, i, i, i, f, p]),
        "gqa_decode_prepared": (i, [p, p, p, p, i, i, i, f, i, p, sz, p]),
        "gqa_decode_fp8kv": (i, [p, p, p, p, i, i, f, f, f, i, p, sz, p]),
        "gqa_decode_split_stage": (i, [p, i, p, i, p, p, i, i, f, f, f, i, p, sz, p]),
        "gqa_decode_combine_stage": (i, [p, p, i, i, i, i, f, i, p, sz, p]),
        "gqa_decode_workspace_init": (i, [p, sz, p]),
        "gqa_decode_get_status": (i, [p, sz, p, ctypes.POINTER(ctypes.c_uint32)]),
        "gqa_decode_noalloc": (i, [p, p, p, p, i, i, i, f, i, p]),
        "gqa_decode_noalloc_get_status": (i, [p, ctypes.POINTER(ctypes.c_uint32)]),
        "gqa_decode_int8kv": (i, [p, p, p, p, p, i, i, i, f, i, p, sz, p]),
        "gqa_decode_paged": (i, [p, i, p, i, p, p, i, i, i, p, p, i, i, f, f, f, i, p, sz, p]),
        "gqa_decode_verify": (i, [p, i, p, i, p, p, p, i, i, i, f, f, f, i, p, sz, p]),
        "gqa_append_kv": (i, [p, p, p, p, p, i, p, p, i, p, p, i, p, i, f, f, f, f, p, sz, p]),
        "gqa_append_kv_paged": (i, [p, p, p, p, p, i, p, p, i, p, p, i, p, p, i, i, i, f, f, f, f, p, sz, p]),
        "gqa_decode_debug_skip_tile": (i, [p, i, p, i, p, p, i, i, f, f, f, i, p, sz, i,
                                           ctypes.c_uint64, p]),
        "gqa_decode_debug_cut_extents": (i, [ctypes.c_uint64, ctypes.c_uint64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None):
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            path = path or LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = _declare(ctypes.CDLL(path))
            if path != LIB_PATH:
                return lib
            _lib = lib
        return _lib


def check(status: int) -> None:
    if status != 0:
        lib = load()
        raise GqaError(status, lib.gqa_status_string(status).decode(),
                       lib.gqa_last_error().decode())
