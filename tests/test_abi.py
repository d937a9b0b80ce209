"""CPU tests of the C-ABI boundary: the library builds for sm_103a, loads without a GPU,
exports exactly what include/bf16delta.h and include/bf16delta_debug.h declare, and its host-only logic (size bounds,
workspace sizes, header parsing, argument checks) behaves as documented.  No call here
launches GPU work."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from lossless_bf16_weight_old_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("bf16delta.h", "bf16delta_debug.h")]


def _declared() -> set[str]:
    src = "".join(open(h).read() for h in HEADERS)
    return set(re.findall(r"^BD_API\s+[\w\s\*]*?\b(bd_\w+)\s*\(", src, flags=re.M))


def test_headers_are_all_listed():
    inc = os.path.join(ROOT, "include")
    assert sorted(os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")) == \
        sorted(HEADERS)


def test_library_exports_every_declared_symbol(cuda_lib):
    names = _declared()
    assert len(names) == 18
    for name in names:
        assert hasattr(cuda_lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.split()[-1].startswith("bd_")}
    assert exported == names


def test_python_signatures_cover_header():
    assert set(_lib.SIGNATURES) == _declared()


def test_compress_bound_is_an_upper_bound(cuda_lib):
    rng = np.random.default_rng(3)
    for n in (0, 1, 7, 24, 4095, 4096, 4097, 20000):
        old = rng.integers(0, 1 << 16, n).astype(np.uint16)
        # worst cases: every element rare; and a mantissa/rare mix near the list/bitmap edge
        cases = [old ^ np.uint16(0x8000), old ^ rng.integers(1, 1 << 16, n).astype(np.uint16)]
        mix = old.copy()
        mix[: n // 20] ^= np.uint16(0x0001)
        mix[n // 20:] ^= np.uint16(0x0080)
        cases.append(mix)
        bound = cuda_lib.bd_compress_bound(n)
        for new in cases:
            payload, _ = oracle.encode(old, new)
            assert payload.size <= bound
            payload2, _ = oracle.encode(old, new, base=12345)   # version 2: 16 bytes longer
            assert payload2.size == payload.size + 16 <= bound
    assert cuda_lib.bd_compress_bound((1 << 40) + 1) == 0


def test_workspace_sizes(cuda_lib):
    def ws(fn, ns):
        arr = (ctypes.c_uint64 * max(1, len(ns)))(*ns)
        return fn(arr, len(ns))
    a = ws(cuda_lib.bd_compress_workspace_size, [1 << 20])
    b = ws(cuda_lib.bd_compress_workspace_size, [1 << 21])
    assert 0 < a < b
    assert a % 256 == 0
    # O(chunks) scratch: compress a 1 KiB slot plus ~30 bytes per 4096-element chunk,
    # decompress ~24 bytes per chunk
    d = ws(cuda_lib.bd_decompress_workspace_size, [1 << 24])
    c = ws(cuda_lib.bd_compress_workspace_size, [1 << 24])
    chunks = (1 << 24) // 4096
    assert 16 * chunks < d <= 32 * chunks + 4096
    assert 1024 * chunks < c <= 1100 * chunks + 4096
    assert ws(cuda_lib.bd_compress_workspace_size, [(1 << 40) + 1]) == 0
    assert ws(cuda_lib.bd_decompress_workspace_size, [1, 2, 3]) > 0


def test_payload_info_parses_oracle_headers(cuda_lib):
    rng = np.random.default_rng(9)
    old = rng.integers(0, 1 << 16, 10000).astype(np.uint16)
    new = old.copy()
    new[::50] ^= np.uint16(3)
    new[7::400] ^= np.uint16(0x4000)
    payload, _ = oracle.encode(old, new)
    info = _lib.PayloadInfo()
    hdr = (ctypes.c_uint8 * 64).from_buffer_copy(payload[:64].tobytes())
    assert cuda_lib.bd_payload_info(hdr, 64, ctypes.byref(info)) == 0
    assert info.n == 10000 and info.chunks == 3 and info.version == 1
    assert info.chunk_elems == 4096 and info.total_size == payload.size
    assert info.n_mant == 200 and info.n_rare == 25
    # flips that break a checked relation (n -> n + 65536 changes C; M, R, size change total)
    for off in (0, 8, 12, 18, 24, 32, 40, 48, 56):
        bad = bytearray(payload[:64].tobytes())
        bad[off] ^= 1
        b = (ctypes.c_uint8 * 64).from_buffer_copy(bytes(bad))
        assert cuda_lib.bd_payload_info(b, 64, ctypes.byref(info)) == 3, off
    assert cuda_lib.bd_payload_info(hdr, 63, ctypes.byref(info)) == 1


def test_payload_info_parses_version_2_headers(cuda_lib):
    rng = np.random.default_rng(10)
    old = rng.integers(0, 1 << 16, 9000).astype(np.uint16)
    new = old.copy()
    new[::30] ^= np.uint16(5)
    base = 0xFEDCBA9876543210
    payload, _ = oracle.encode(old, new, base=base)
    info = _lib.PayloadInfo()
    hdr = (ctypes.c_uint8 * 80).from_buffer_copy(payload[:80].tobytes())
    assert cuda_lib.bd_payload_info(hdr, 80, ctypes.byref(info)) == 0
    assert info.version == 2 and info.base_checksum == base
    assert info.n == 9000 and info.total_size == payload.size
    # a version-2 header needs all 80 bytes; the reserved word must be zero
    assert cuda_lib.bd_payload_info(hdr, 64, ctypes.byref(info)) == 1
    bad = bytearray(payload[:80].tobytes())
    bad[75] = 1
    b = (ctypes.c_uint8 * 80).from_buffer_copy(bytes(bad))
    assert cuda_lib.bd_payload_info(b, 80, ctypes.byref(info)) == 3
    # a version-1 header reports base 0
    p1, _ = oracle.encode(old, new)
    h1 = (ctypes.c_uint8 * 64).from_buffer_copy(p1[:64].tobytes())
    assert cuda_lib.bd_payload_info(h1, 64, ctypes.byref(info)) == 0
    assert info.version == 1 and info.base_checksum == 0


def test_payload_info_parses_version_3_headers(cuda_lib):
    rng = np.random.default_rng(12)
    old = rng.integers(0, 1 << 16, 7 * 4096 + 7).astype(np.uint16)
    new = old.copy()
    new[:5 * 4096:40] ^= np.uint16(3)                   # compact chunks
    new[3 * 4096:5 * 4096:1500] ^= np.uint16(0x4001)
    new[5 * 4096 + 600:6 * 4096:10] ^= np.uint16(5)     # compact, first gap escaped
    base = 0x0102030405060708
    payload, _ = oracle.encode(old, new, base=base, compact=True)
    C = 8
    table = payload[80:80 + 4 * C].view(np.uint32)
    compact = (table >> 31) == 1
    n_esc = int(np.where(compact, (table >> 18) & 0x1FF, 0).sum())
    assert compact.any() and (~compact).any() and n_esc > 0
    info = _lib.PayloadInfo()
    hdr = (ctypes.c_uint8 * 80).from_buffer_copy(payload[:80].tobytes())
    assert cuda_lib.bd_payload_info(hdr, 80, ctypes.byref(info)) == 0
    assert info.version == 3 and info.base_checksum == base and info.n_escapes == n_esc
    assert info.total_size == payload.size and info.chunks == C
    # a total that leaves an odd number of bytes (or fewer than the other sections) is refused
    for delta in (1, -2 * n_esc - 2):
        bad = bytearray(payload[:80].tobytes())
        bad[56:64] = (payload.size + delta).to_bytes(8, "little")
        b = (ctypes.c_uint8 * 80).from_buffer_copy(bytes(bad))
        assert cuda_lib.bd_payload_info(b, 80, ctypes.byref(info)) == 3, delta
    # version 2 and 1 report no escapes
    p2, _ = oracle.encode(old, new, base=base)
    h2 = (ctypes.c_uint8 * 80).from_buffer_copy(p2[:80].tobytes())
    assert cuda_lib.bd_payload_info(h2, 80, ctypes.byref(info)) == 0
    assert info.version == 2 and info.n_escapes == 0 and info.flags == 0


def test_payload_info_reports_overwrite_flag(cuda_lib):
    rng = np.random.default_rng(14)
    old = rng.integers(0, 1 << 16, 6000).astype(np.uint16)
    new = old.copy()
    new[::25] ^= np.uint16(9)
    info = _lib.PayloadInfo()
    for compact in (False, True):
        p, _ = oracle.encode(old, new, base=77, compact=compact, overwrite=True)
        h = (ctypes.c_uint8 * 80).from_buffer_copy(p[:80].tobytes())
        assert cuda_lib.bd_payload_info(h, 80, ctypes.byref(info)) == 0
        assert info.flags == 1 and info.version == (3 if compact else 2)
        bad = bytearray(p[:80].tobytes())
        bad[72] = 3
        b = (ctypes.c_uint8 * 80).from_buffer_copy(bytes(bad))
        assert cuda_lib.bd_payload_info(b, 80, ctypes.byref(info)) == 3


def test_payload_info_parses_version_4_headers(cuda_lib):
    rng = np.random.default_rng(15)
    old = rng.integers(0, 1 << 16, 5 * 4096 + 9).astype(np.uint16)
    new = old.copy()
    new[:3 * 4096:37] ^= np.uint16(3)
    new[4096:2 * 4096:700] ^= np.uint16(0x8001)
    info = _lib.PayloadInfo()
    for ow in (False, True):
        p, _ = oracle.encode(old, new, base=99, rice=True, overwrite=ow)
        table = p[80:80 + 4 * 6].view(np.uint32)
        assert ((table >> 31) == 1).any()
        h = (ctypes.c_uint8 * 80).from_buffer_copy(p[:80].tobytes())
        assert cuda_lib.bd_payload_info(h, 80, ctypes.byref(info)) == 0
        assert info.version == 4 and info.base_checksum == 99 and info.n_escapes == 0
        assert info.total_size == p.size and info.flags == int(ow)
        # no X stream: the total is exactly the sections
        bad = bytearray(p[:80].tobytes())
        bad[56:64] = (p.size + 2).to_bytes(8, "little")
        b = (ctypes.c_uint8 * 80).from_buffer_copy(bytes(bad))
        assert cuda_lib.bd_payload_info(b, 80, ctypes.byref(info)) == 3
    bad = bytearray(p[:80].tobytes())
    bad[8] = 5
    b = (ctypes.c_uint8 * 80).from_buffer_copy(bytes(bad))
    assert cuda_lib.bd_payload_info(b, 80, ctypes.byref(info)) == 3


def test_version_3_bound(cuda_lib):
    """bd_compress_bound covers versions 3 and 4: never longer than version 2 of the same
    update."""
    rng = np.random.default_rng(13)
    for n in (1, 4097, 3 * 4096 + 5):
        old = rng.integers(0, 1 << 16, n).astype(np.uint16)
        for rate in (0.001, 0.05, 0.5, 1.0):
            new = old ^ np.where(rng.random(n) < rate, rng.integers(1, 1 << 16, n), 0).astype(np.uint16)
            p3, _ = oracle.encode(old, new, base=1, compact=True)
            p4, _ = oracle.encode(old, new, base=1, rice=True)
            p2, _ = oracle.encode(old, new, base=1)
            assert max(p3.size, p4.size) <= p2.size <= cuda_lib.bd_compress_bound(n)


def test_argument_checks_need_no_gpu(cuda_lib):
    """Bad arguments are rejected before any CUDA call."""
    one = ctypes.c_uint64(1)
    dummy = ctypes.c_void_p(4096)
    # null tensors
    assert cuda_lib.bd_compress(None, None, 10, dummy, 100, dummy, 1 << 20, dummy, dummy,
                                None, None) == 1
    # misaligned tensor
    assert cuda_lib.bd_compress(ctypes.c_void_p(4098), dummy, 10, ctypes.c_void_p(1 << 20),
                                100, dummy, 1 << 20, dummy, dummy, None, None) == 1
    # workspace too small
    assert cuda_lib.bd_compress(dummy, dummy, 10, ctypes.c_void_p(1 << 20), 100,
                                ctypes.c_void_p(1 << 24), 16, dummy, dummy, None, None) == 1
    # decompress needs a status word and an expected checksum
    assert cuda_lib.bd_decompress(dummy, 10, dummy, 100, dummy, dummy, dummy, 1 << 20, None,
                                  None) == 1
    # partially overlapping out-of-place output
    assert cuda_lib.bd_decompress(ctypes.c_void_p(1 << 20), 1000, ctypes.c_void_p(1 << 24),
                                  100, dummy, ctypes.c_void_p((1 << 20) + 16),
                                  ctypes.c_void_p(1 << 26), 1 << 20, dummy, None) == 1
    # the versioned compress takes format 2, 3 or 4 only, optionally with the overwrite bit
    for fmt in (0, 1, 5, 0x102 | 0x200, 0x101, 0x105):
        assert cuda_lib.bd_compress_versioned(dummy, dummy, 10, ctypes.c_void_p(1 << 20), 100,
                                              ctypes.c_void_p(1 << 24), 1 << 20, dummy, dummy,
                                              dummy, fmt, None, None) == 1
    base_ptrs = (ctypes.c_void_p * 1)(4096)
    assert cuda_lib.bd_compress_versioned_batch(None, base_ptrs, 0, 7, ctypes.c_void_p(1 << 24),
                                                1 << 20, None, None) == 1
    assert cuda_lib.bd_checksum(None, 5, dummy, None) == 1
    # the no-workspace apply: an expected checksum or status word off its alignment, a missing
    # status word and a tensor beyond its scratch are rejected before anything is enqueued
    base = 1 << 20
    for exp, st in ((ctypes.c_void_p(base + 4), dummy), (dummy, ctypes.c_void_p(base + 2)),
                    (dummy, None), (None, dummy)):
        assert cuda_lib.bd_decompress_noalloc(ctypes.c_void_p(1 << 24), 4096,
                                              ctypes.c_void_p(1 << 26), 64, exp,
                                              ctypes.c_void_p(1 << 24), st, None) == 1
    assert cuda_lib.bd_decompress_noalloc(dummy, (1 << 27) + 1, dummy, 64, dummy, dummy, dummy,
                                          None) == 1
    assert cuda_lib.bd_status_sync(None, None) == 1
    # the streamed apply: every argument is checked before anything is enqueued
    it = (_lib.DecompressItem * 1)()
    it[0].d_old = it[0].d_out = 1 << 24
    it[0].n = 4096
    it[0].d_payload = 1 << 12   # (a host address; never read here)
    it[0].size = 1000
    it[0].d_expected = 4096
    ws, stg, st = ctypes.c_void_p(1 << 28), ctypes.c_void_p(1 << 30), ctypes.c_void_p(1 << 26)
    s1, s2 = ctypes.c_void_p(0x5000), ctypes.c_void_p(0x6000)
    streamed = cuda_lib.bd_decompress_batch_streamed
    assert streamed(it, 1, stg, 1024, ws, 1 << 20, st, s1, None) == 1      # no copy stream
    assert streamed(it, 1, stg, 1024, ws, 1 << 20, st, s1, s1) == 1        # the same stream
    assert streamed(it, 1, stg, 768, ws, 1 << 20, st, s1, s2) == 1         # payload > slot
    assert streamed(it, 1, stg, 1000, ws, 1 << 20, st, s1, s2) == 1        # slot not 256k
    assert streamed(it, 1, stg, 1 << 62, ws, 1 << 20, st, s1, s2) == 1     # slot too large
    assert streamed(it, 1, ctypes.c_void_p((1 << 30) + 16), 1024, ws, 1 << 20, st, s1,
                    s2) == 1                                                 # staging alignment
    assert streamed(it, 1, ctypes.c_void_p((1 << 24) + 4096), 1024, ws, 1 << 20, st, s1,
                    s2) == 1                                                 # staging over out
    assert streamed(it, 1, stg, 1024, ws, 16, st, s1, s2) == 1              # workspace too small
    assert streamed(it, 1, stg, 1024, ws, 1 << 20, None, s1, s2) == 1      # no status word
    it[0].d_payload = None
    assert streamed(it, 1, stg, 1024, ws, 1 << 20, st, s1, s2) == 1        # no payload
    # the fault-injection hook stalls a tensor of the call, no other
    items = (_lib.CompressItem * 2)()
    for stall in (2, 3, 1 << 31):
        assert cuda_lib.bd_debug_compress_stall(items, 2, stall, ctypes.c_void_p(1 << 24),
                                                1 << 20, None, None) == 1
    assert cuda_lib.bd_debug_compress_stall(None, 0, 0, ctypes.c_void_p(1 << 24), 1 << 20,
                                            None, None) == 1
    del one


def test_status_strings(cuda_lib):
    for code, word in [(0, b"ok"), (2, b"capacity"), (3, b"malformed"), (4, b"checksum")]:
        assert word in cuda_lib.bd_status_string(code)


def test_build_targets_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)
