"""ctypes loader for libpagedkv.so: declares the C ABI of include/pagedkv.h.

There is no fallback: if the library is missing the first call raises.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

# pkv_dtype
F32 = 0
BF16 = 1

# pkv_status
OK = 0
EINVAL = -1
EUNSUPPORTED = -2
EALIGN = -3
ECUDA = -4
EWORKSPACE = -5
ESCRATCH = -6

NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

# device error word bits
DERR_SLOT_RANGE = 0x1
DERR_BLOCK_RANGE = 0x2
DERR_LEN_RANGE = 0x4
DERR_WAIT_TIMEOUT = 0x8

# (name, restype, argtypes) of every exported symbol
_P = ctypes.c_void_p
_I = ctypes.c_int32
_F = ctypes.c_float
_S = ctypes.c_size_t
SIGNATURES = [
    ("pkv_version", ctypes.c_int, []),
    ("pkv_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("pkv_get_device_error", ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    ("pkv_kv_store", ctypes.c_int, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_int, _P]),
    ("pkv_paged_decode_workspace_bytes", _S, [_I, _I, _I, _I]),
    ("pkv_paged_decode_attn", ctypes.c_int,
     [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, ctypes.c_int, _P]),
    ("pkv_copy_blocks", ctypes.c_int,
     [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), _I, _P, _I, _I, ctypes.c_int64, _P]),
    ("pkv_kv_store_fp8", ctypes.c_int, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _P]),
    ("pkv_paged_decode_attn_fp8", ctypes.c_int,
     [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _I, _P, _S, _P]),
    ("pkv_paged_verify_attn", ctypes.c_int,
     [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, ctypes.c_int, _P]),
    ("pkv_paged_decode_attn_noalloc", ctypes.c_int,
     [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, ctypes.c_int, _P]),
    ("pkv_paged_varlen_prefill_attn", ctypes.c_int,
     [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S,
      ctypes.c_int, _P]),
    ("pkv_paged_varlen_prefill_workspace_bytes", _S, [_I, _I, _I, _I, _I]),
]

_lib = None


class LibraryMissing(RuntimeError):
    pass


def load() -> ctypes.CDLL:
    """Load the library once; raise if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryMissing(
            f"{LIB_PATH} is missing: build it with `python -m pagedattention_kv_cache_gb300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, restype, argtypes in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = restype
        fn.argtypes = argtypes
    _lib = lib
    return lib


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = load().pkv_status_string(status).decode()
        super().__init__(f"{fn} failed: {msg} (status {status})")


def check(fn: str, status: int) -> None:
    if status != OK:
        raise PagedKVError(fn, status)
