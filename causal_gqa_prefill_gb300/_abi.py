"""ctypes binding of the C ABI declared in include/attn_prefill.h.

Argument marshalling only: every step of the attention passes runs in the
CUDA library. There is no CPU fallback; a missing library raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_CHECK = 5

# Every function the public header declares, with its ctypes signature.
_SIGNATURES = {
    "attn_prefill_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_float, ctypes.c_void_p]),
    "attn_prefill_fwd_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_float, ctypes.c_void_p]),
    "attn_prefill_fwd_chunk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_float, ctypes.c_void_p]),
    "attn_prefill_fwd_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_float, ctypes.c_float,
                                            ctypes.c_float, ctypes.c_float, ctypes.c_void_p]),
    "attn_decode_workspace_bytes": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64,
                                                     ctypes.c_int32, ctypes.c_int32,
                                                     ctypes.c_int32]),
    "attn_decode_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_float, ctypes.c_void_p]),
    "attn_prefill_bwd_workspace_bytes": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64,
                                                          ctypes.c_int32, ctypes.c_int32,
                                                          ctypes.c_int32]),
    "attn_prefill_bwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_float, ctypes.c_void_p]),
    "attn_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p]),
    "attn_selftest_wait_timeout_noalloc": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p]),
    "attn_prefill_host_staging_bytes": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64,
                                                         ctypes.c_int64, ctypes.c_int32,
                                                         ctypes.c_int32, ctypes.c_int32]),
    "attn_prefill_fwd_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                             ctypes.c_void_p]),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_debug_check_count": (ctypes.c_int64, []),
    "attn_device_check": (ctypes.c_int, [ctypes.c_void_p]),
    "attn_prefill_grid_size": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.library_path()


def load(path: str | None = None):
    """Load (once) and return the ctypes handle of the CUDA library."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library not built ({p} missing); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()
