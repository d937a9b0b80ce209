"""CPU oracle of the BF16DLT1 delta format -- TEST INFRASTRUCTURE ONLY.

A plain single-threaded C implementation (``bd_oracle.c``) of what the delta path computes,
wrapped with ctypes for numpy arrays.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) may import this package.
The CUDA library never imports, links or executes anything here, and this package imports
nothing from the library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bd_oracle.c")
_LIB = os.path.join(_HERE, "libbd_oracle.so")

OK, ERR_ARG, ERR_CAPACITY, ERR_FORMAT, ERR_CHECKSUM = 0, 1, 2, 3, 4
ERR_BASE = 6

_lib = None


def build(force: bool = False) -> str:
    """Compiles bd_oracle.c into libbd_oracle.so next to it (plain gcc, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", tmp, _SRC],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, p = ctypes.c_uint64, ctypes.c_void_p
        lib.orc_checksum.argtypes = [p, u64]
        lib.orc_checksum.restype = u64
        lib.orc_encode.argtypes = [p, p, u64, p, u64, ctypes.POINTER(u64), ctypes.POINTER(u64)]
        lib.orc_encode.restype = ctypes.c_int
        lib.orc_encode_versioned.argtypes = [p, p, u64, u64, p, u64, ctypes.POINTER(u64),
                                             ctypes.POINTER(u64)]
        lib.orc_encode_versioned.restype = ctypes.c_int
        lib.orc_encode_compact.argtypes = [p, p, u64, u64, p, u64, ctypes.POINTER(u64),
                                           ctypes.POINTER(u64)]
        lib.orc_encode_compact.restype = ctypes.c_int
        for name in ("orc_encode_overwrite", "orc_encode_compact_overwrite"):
            fn = getattr(lib, name)
            fn.argtypes = [p, p, u64, u64, p, u64, ctypes.POINTER(u64), ctypes.POINTER(u64)]
            fn.restype = ctypes.c_int
        lib.orc_encode_rice.argtypes = [p, p, u64, u64, ctypes.c_int, p, u64,
                                        ctypes.POINTER(u64), ctypes.POINTER(u64)]
        lib.orc_encode_rice.restype = ctypes.c_int
        lib.orc_decode.argtypes = [p, u64, p, u64, u64, p]
        lib.orc_decode.restype = ctypes.c_int
        lib.orc_decode_incremental.argtypes = [p, u64, p, u64, u64, u64, p,
                                               ctypes.POINTER(u64)]
        lib.orc_decode_incremental.restype = ctypes.c_int
        _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype.itemsize == 2 else a.astype(np.uint16)
    return a.reshape(-1)


def checksum(w) -> int:
    """Checksum of a BF16 tensor given as any 16-bit numpy array."""
    w = _u16(w)
    return int(_load().orc_checksum(w.ctypes.data, w.size))


def encode(old, new, base: int | None = None, compact: bool = False,
           overwrite: bool = False, rice: bool = False,
           cap: int | None = None) -> tuple[np.ndarray, int]:
    """Returns (payload bytes as a uint8 array, checksum of new).  With `base` (the checksum of
    old as the caller knows it) the payload is version 2, bound to that base; with compact=True
    (which needs a base) it is version 3, with compact position lists; with rice=True (which
    needs a base, and excludes compact) it is version 4, with Rice-coded compact position
    blocks; with overwrite=True (which needs a base) its streams hold new values instead of XOR
    masks.  `cap` only saves time: when given, the encoder first writes into a buffer of that
    many bytes in one pass and is run again with the exact size only if the payload is
    larger; the result is the same either way."""
    old, new = _u16(old), _u16(new)
    if old.size != new.size:
        raise ValueError("old and new must have the same number of elements")
    lib = _load()
    size, ck = ctypes.c_uint64(), ctypes.c_uint64()
    if (compact or overwrite or rice) and base is None:
        raise ValueError("compact, Rice and overwrite payloads are bound to a base: give base")
    if compact and rice:
        raise ValueError("compact (version 3) and rice (version 4) exclude each other")
    if rice:
        b = ctypes.c_uint64(int(base) & (2**64 - 1))
        call = lambda out, cap: lib.orc_encode_rice(old.ctypes.data, new.ctypes.data, old.size, b,
                                                    int(bool(overwrite)), out, cap,
                                                    ctypes.byref(size), ctypes.byref(ck))
    elif base is None:
        call = lambda out, cap: lib.orc_encode(old.ctypes.data, new.ctypes.data, old.size, out,
                                               cap, ctypes.byref(size), ctypes.byref(ck))
    else:
        b = ctypes.c_uint64(int(base) & (2**64 - 1))
        fn = {(False, False): lib.orc_encode_versioned, (True, False): lib.orc_encode_compact,
              (False, True): lib.orc_encode_overwrite,
              (True, True): lib.orc_encode_compact_overwrite}[(bool(compact), bool(overwrite))]
        call = lambda out, cap: fn(old.ctypes.data, new.ctypes.data, old.size, b, out, cap,
                                   ctypes.byref(size), ctypes.byref(ck))
    if cap is not None:
        out = np.zeros(max(int(cap), 1), dtype=np.uint8)
        rc = call(out.ctypes.data, out.size)
        if rc == OK:
            return out[:size.value].copy(), int(ck.value)
        if rc != ERR_CAPACITY:
            raise RuntimeError(f"orc_encode failed with {rc}")
    else:
        rc = call(None, 0)
        if rc not in (OK, ERR_CAPACITY):
            raise RuntimeError(f"orc_encode failed with {rc}")
    out = np.zeros(size.value, dtype=np.uint8)
    rc = call(out.ctypes.data, out.size)
    if rc != OK:
        raise RuntimeError(f"orc_encode failed with {rc}")
    return out, int(ck.value)


def decode(old, payload, expected_checksum: int) -> tuple[int, np.ndarray]:
    """Returns (status, restored).  status is OK, ERR_FORMAT or ERR_CHECKSUM."""
    old = _u16(old)
    payload = np.ascontiguousarray(payload, dtype=np.uint8).reshape(-1)
    out = np.empty_like(old)
    rc = _load().orc_decode(old.ctypes.data, old.size, payload.ctypes.data, payload.size,
                            ctypes.c_uint64(expected_checksum & (2**64 - 1)),
                            out.ctypes.data)
    return int(rc), out


def decode_incremental(old, payload, ck_old: int, expected_checksum: int
                       ) -> tuple[int, np.ndarray, int]:
    """Incremental verification: returns (status, restored, ck) where ck = ck_old plus the
    new-minus-old checksum terms of the changed words (ck is 0 when the payload is
    malformed)."""
    old = _u16(old)
    payload = np.ascontiguousarray(payload, dtype=np.uint8).reshape(-1)
    out = np.empty_like(old)
    ck = ctypes.c_uint64(0)
    rc = _load().orc_decode_incremental(old.ctypes.data, old.size, payload.ctypes.data,
                                        payload.size, ctypes.c_uint64(ck_old & (2**64 - 1)),
                                        ctypes.c_uint64(expected_checksum & (2**64 - 1)),
                                        out.ctypes.data, ctypes.byref(ck))
    return int(rc), out, int(ck.value)
