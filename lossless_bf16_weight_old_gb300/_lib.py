"""ctypes loader of libbf16delta.so (argument types only; no computation here).

The library is built in-tree by ``build.py``.  There is no fallback: if the shared library is
missing and cannot be built, loading fails with an error.
"""
from __future__ import annotations

import ctypes

from . import build as _build

c_u64, c_u32, c_int, c_p = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p


class CompressItem(ctypes.Structure):
    _fields_ = [("d_old", c_p), ("d_new", c_p), ("n", c_u64), ("d_payload", c_p),
                ("cap", c_u64), ("d_size", c_p), ("d_checksum", c_p), ("d_status", c_p)]


class DecompressItem(ctypes.Structure):
    _fields_ = [("d_old", c_p), ("d_out", c_p), ("n", c_u64), ("d_payload", c_p),
                ("size", c_u64), ("d_expected", c_p), ("d_status", c_p)]


class IncrementalItem(ctypes.Structure):
    _fields_ = [("d_w", c_p), ("n", c_u64), ("d_payload", c_p), ("size", c_u64),
                ("d_ck_old", c_p), ("d_expected", c_p), ("d_ck_out", c_p), ("d_status", c_p)]


class PayloadInfo(ctypes.Structure):
    _fields_ = [("n", c_u64), ("chunks", c_u64), ("n_mant", c_u64), ("n_rare", c_u64),
                ("position_bytes", c_u64), ("total_size", c_u64), ("version", c_u32),
                ("chunk_elems", c_u32), ("base_checksum", c_u64), ("n_escapes", c_u64),
                ("flags", c_u64)]


# name -> (restype, argtypes); must match include/bf16delta.h and include/bf16delta_debug.h
SIGNATURES = {
    "bd_compress_bound": (c_u64, [c_u64]),
    "bd_compress_workspace_size": (c_u64, [c_p, c_u32]),
    "bd_decompress_workspace_size": (c_u64, [c_p, c_u32]),
    "bd_compress": (c_int, [c_p, c_p, c_u64, c_p, c_u64, c_p, c_u64, c_p, c_p, c_p, c_p]),
    "bd_compress_batch": (c_int, [c_p, c_u32, c_p, c_u64, c_p, c_p]),
    "bd_compress_versioned": (c_int, [c_p, c_p, c_u64, c_p, c_u64, c_p, c_u64, c_p, c_p, c_p, c_u32,
                                      c_p, c_p]),
    "bd_compress_versioned_batch": (c_int, [c_p, c_p, c_u32, c_u32, c_p, c_u64, c_p, c_p]),
    "bd_decompress": (c_int, [c_p, c_u64, c_p, c_u64, c_p, c_p, c_p, c_u64, c_p, c_p]),
    "bd_decompress_batch": (c_int, [c_p, c_u32, c_p, c_u64, c_p, c_p]),
    "bd_decompress_batch_streamed": (c_int, [c_p, c_u32, c_p, c_u64, c_p, c_u64, c_p, c_p, c_p]),
    "bd_decompress_noalloc": (c_int, [c_p, c_u64, c_p, c_u64, c_p, c_p, c_p, c_p]),
    "bd_decompress_incremental": (c_int, [c_p, c_u64, c_p, c_u64, c_p, c_p, c_p, c_p, c_u64, c_p,
                                          c_p]),
    "bd_decompress_incremental_batch": (c_int, [c_p, c_u32, c_p, c_u64, c_p, c_p]),
    "bd_checksum": (c_int, [c_p, c_u64, c_p, c_p]),
    "bd_payload_info": (c_int, [c_p, c_u64, ctypes.POINTER(PayloadInfo)]),
    "bd_status_sync": (c_int, [c_p, c_p]),
    "bd_status_string": (ctypes.c_char_p, [c_int]),
    "bd_debug_compress_stall": (c_int, [c_p, c_u32, c_u32, c_p, c_u64, c_p, c_p]),
}

_lib = None


def path() -> str:
    return _build.LIB


def load():
    """Returns the loaded library, building it first when it is missing or stale."""
    global _lib
    if _lib is None:
        if not _build.up_to_date():
            try:
                _build.build()
            except Exception as e:  # no fallback path exists
                raise RuntimeError(f"libbf16delta.so is missing and could not be built: {e}") from e
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
