"""ctypes view of libmla_decode.so (the C ABI in include/mla_decode.h)."""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

c_int32, c_uint32, c_size_t, c_void_p, c_float = (ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t,
                                                  ctypes.c_void_p, ctypes.c_float)

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE_TOO_SMALL = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_CHECK = 5
MLA_ERR_TIMEOUT = 6

MLA_MASK_NULL = 0
MLA_MASK_CAUSAL = 1
MLA_MASK_SLIDING_WINDOW_CAUSAL = 2
MLA_FLAG_DEBUG_CHECKS = 1
MLA_FLAG_KERNEL_TIMING = 2
MLA_FLAG_FOLD_PAIRS = 4
MLA_FLAG_PER_TOKEN = 8
KERNEL_NAMES = ("absorb_w_uk", "decode_splitkv", "w_uv")

EXPORTED = ("mla_decode_workspace_size", "mla_decode_paged", "mla_decode_paged_fp8",
            "mla_decode_sparse", "mla_decode_kernel_times", "mla_branch_prologue",
            "mla_indexer_workspace_size", "mla_indexer_fp8",
            "mla_debug_wait_selftest",
            "mla_status_string")


class MlaDims(ctypes.Structure):
    _fields_ = [("num_heads", c_int32), ("qk_nope", c_int32), ("qk_rope", c_int32),
                ("kv_lora_rank", c_int32), ("v_head", c_int32), ("page_size", c_int32),
                ("num_pages", c_int32)]


class MlaOpts(ctypes.Structure):
    _fields_ = [("mask", c_int32), ("window", c_int32), ("scale", c_float),
                ("num_splits", c_int32), ("flags", c_uint32)]


_P = ctypes.POINTER
_SIGS = {
    "mla_decode_workspace_size": [_P(MlaDims), _P(MlaOpts), c_int32, c_int32, _P(c_size_t)],
    "mla_decode_paged": [_P(MlaDims), _P(MlaOpts), c_void_p, c_void_p, c_int32, c_int32, c_void_p,
                         c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                         c_void_p, c_size_t, c_void_p],
    "mla_decode_paged_fp8": [_P(MlaDims), _P(MlaOpts), c_void_p, c_void_p, c_int32, c_int32,
                             c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                             c_void_p],
    "mla_decode_sparse": [_P(MlaDims), _P(MlaOpts), c_void_p, c_void_p, c_int32, c_int32, c_void_p,
                          c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                          c_void_p, c_size_t, c_void_p],
    "mla_debug_wait_selftest": [ctypes.c_uint64, c_void_p, c_size_t, c_void_p],
    "mla_indexer_workspace_size": [c_int32, c_int32, c_int32, c_int32, c_int32, _P(c_size_t)],
    "mla_indexer_fp8": [c_int32, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_int32,
                        c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_int32,
                        c_int32, c_void_p, c_void_p, c_uint32, c_void_p, c_size_t, c_void_p],
    "mla_branch_prologue": [_P(MlaDims), c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p,
                            c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_float, c_uint32,
                            c_void_p, c_size_t, c_void_p],
}

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load the in-tree library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"{LIB} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(LIB)
            for name, args in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.mla_decode_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_float), c_int32]
            lib.mla_decode_kernel_times.restype = ctypes.c_int
            lib.mla_status_string.argtypes = [ctypes.c_int]
            lib.mla_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().mla_status_string(code).decode()


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({status_string(code)})")
        self.code = code


def kernel_times():
    """Mean per-kernel durations (ms) over the calls made with MLA_FLAG_KERNEL_TIMING since
    the previous read, and the number of calls they average."""
    buf = (ctypes.c_float * len(KERNEL_NAMES))()
    n = load().mla_decode_kernel_times(buf, len(KERNEL_NAMES))
    if n < 0:
        raise RuntimeError("mla_decode_kernel_times failed")
    return (dict(zip(KERNEL_NAMES, list(buf))) if n > 0 else {}), n
