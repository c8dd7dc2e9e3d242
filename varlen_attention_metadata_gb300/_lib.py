"""ctypes declarations of the libpseq.so C ABI (``include/pseq.h``).

Argument marshalling only: every function here is the C entry point of the
same name.  The library is loaded from this package's directory; when it is
missing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpseq.so")

PSEQ_OK = 0
PSEQ_ERR_ARG = 1
PSEQ_ERR_OVERFLOW = 2
PSEQ_ERR_VALUE = 3
PSEQ_ERR_CAPACITY = 4
PSEQ_ERR_TIMEOUT = 5
PSEQ_ERR_CUDA = 6
STATUS_NAMES = {
    PSEQ_OK: "PSEQ_OK",
    PSEQ_ERR_ARG: "PSEQ_ERR_ARG",
    PSEQ_ERR_OVERFLOW: "PSEQ_ERR_OVERFLOW",
    PSEQ_ERR_VALUE: "PSEQ_ERR_VALUE",
    PSEQ_ERR_CAPACITY: "PSEQ_ERR_CAPACITY",
    PSEQ_ERR_TIMEOUT: "PSEQ_ERR_TIMEOUT",
    PSEQ_ERR_CUDA: "PSEQ_ERR_CUDA",
}
PSEQ_MAX_FIELDS = 8
PSEQ_STATIC_MAX_TOKENS = 1 << 24


class PseqInfo(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int32), ("count", ctypes.c_int32),
                ("max_seqlen", ctypes.c_int32), ("total", ctypes.c_int32)]


class PseqField(ctypes.Structure):
    _fields_ = [("src", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("elem_bytes", ctypes.c_int32),
                ("planes", ctypes.c_int32), ("row_elems", ctypes.c_int64)]


class PseqError(RuntimeError):
    """A libpseq call failed; ``status`` is the pseq_status code."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), in header order
SIGNATURES = {
    "pseq_version": (ctypes.c_int, []),
    "pseq_last_error": (ctypes.c_char_p, []),
    "pseq_launch_count": (_I64, []),
    "pseq_debug_set_wait": (None, [_I64, _I64]),
    "pseq_debug_wait_limit_ns": (_I64, []),
    "pseq_from_doc_ids_workspace_size": (_SZ, [_I64, _I64]),
    "pseq_from_doc_ids": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "pseq_from_doc_ids_static": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _P]),
    "thd_workspace_size": (_SZ, [_I64, _I64]),
    "thd_from_batch": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _I32, _P, _I32,
                                      _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "thd_meta": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "thd_gather": (ctypes.c_int, [_P, _I32, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "thd_padding_mask": (ctypes.c_int, [_I64, _P, _P, _I64, _P, _P, _P, _SZ, _P]),
    "thd_chunks_from_batch": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _I64, _I32, _P, _I32,
                                             _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "thd_mask_from_token_ids_workspace_size": (_SZ, [_I64]),
    "thd_mask_from_token_ids": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _P, _SZ, _P]),
    "pack_ffd": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
    "pseq_doc_ids_to_lengths_workspace_size": (_SZ, [_I64, _I64]),
    "pseq_doc_ids_to_lengths": (ctypes.c_int, [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "pack_squeeze_workspace_size": (_SZ, [_I64, _I64]),
    "pack_squeeze": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, _P, _P, _I64, _I64, _I64, _I64, _I32,
                                    _I64, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]),
}

_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libpseq.so and declare every entry point.  Raises when missing."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libpseq.so not found at {path}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()'); there is no fallback path")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path == LIB_PATH:
            _lib = lib
        return lib


def last_error() -> str:
    msg = load().pseq_last_error()
    return msg.decode() if msg else ""


def check(status: int):
    """Raise PseqError for a non-zero host-side status."""
    if status != PSEQ_OK:
        raise PseqError(status, last_error())
