"""ctypes binding of libdflash_gb300.so: signatures, loading and status codes.

The library is built in-tree from csrc/ (see build.py). Loading fails loudly when it
cannot be built or loaded. There is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

DFLASH_OK = 0
DFLASH_INVALID_ARGUMENT = 1
DFLASH_UNSUPPORTED = 2
DFLASH_WORKSPACE_TOO_SMALL = 3
DFLASH_CUDA_ERROR = 4
DFLASH_NO_DEVICE = 5

DEVICE_BAD_ID = 0x1
DEVICE_TIMEOUT = 0x2

HEADER = os.path.join(_build.ROOT, "include", "dflash.h")

_p, _i, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float

# name -> (restype, argtypes)
SIGNATURES = {
    "dflash_version": (ctypes.c_char_p, []),
    "dflash_status_string": (ctypes.c_char_p, [_i]),
    "dflash_last_error": (ctypes.c_char_p, []),
    "dflash_topk_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "dflash_selector_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "dflash_topk_candidates": (_i, [_p, _i, _i, _i, _i, _f, _f, _p, _p, _p, _sz, _p]),
    "dflash_topk_candidates_noalloc": (_i, [_p, _i, _i, _i, _i, _p, _p, _p]),
    "dflash_lmhead_topk_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "dflash_lmhead_topk": (_i, [_p, _p, _i, _i, _i, _i, _i, _f, _f, _p, _p, _p, _sz, _p]),
    "dflash_hidden_projection": (_i, [_p, _p, _i, _i, _i, _i, _p, _p]),
    "dflash_candidate_edges": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _p, _p]),
    "dflash_selector": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _f, _p, _p,
                             _p, _p, _p, _sz, _p]),
    "dflash_selector_forward": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p,
                                     _p]),
    "dflash_best_path": (_i, [_p, _p, _i, _i, _i, _p, _p, _p, _p]),
    "dflash_selector_lmhead_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "dflash_selector_lmhead": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _f, _p,
                                    _p, _p, _p, _p, _sz, _p]),
    "dflash_device_status": (_i, [ctypes.POINTER(ctypes.c_uint32), _i]),
    "dflash_selftest_wait_timeout": (_i, []),
    "dflash_trace_begin": (_i, [_i]),
    "dflash_trace_end": (_i, [ctypes.POINTER(ctypes.c_float), _i, ctypes.POINTER(ctypes.c_int)]),
}


class DflashError(RuntimeError):
    """A CUDA or device failure reported by the library."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/dflash.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_\w+)\s*\(", text)))


def load(build_if_needed: bool = True):
    """The loaded library (built first if its sources changed)."""
    global _lib
    if _lib is None:
        path = _build.build() if build_if_needed else _build.LIBRARY
        if not os.path.exists(path):
            raise RuntimeError(f"the selector library is missing at {path}; build it with "
                               "draft_candidate_selector_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(status: int) -> None:
    """Raise the exception that matches a non-OK status."""
    if status == DFLASH_OK:
        return
    lib = load()
    name = lib.dflash_status_string(status).decode()
    detail = lib.dflash_last_error().decode()
    msg = f"{name}: {detail}"
    if status in (DFLASH_INVALID_ARGUMENT, DFLASH_WORKSPACE_TOO_SMALL):
        raise ValueError(msg)
    if status == DFLASH_UNSUPPORTED:
        raise NotImplementedError(msg)
    raise DflashError(status, msg)
