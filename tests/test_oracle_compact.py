"""Pins of the oracle's version-3 payloads (compact position lists), CPU only.

Pinned against:
  - one payload worked out by hand from the version-3 layout (below, byte by byte);
  - a bound that follows from the encoder's choice: every chunk is coded compactly only when
    that is smaller, so a version-3 payload is never longer than the version-1 payload plus
    the 16 bytes of the longer header;
  - exact restore, the incremental checksum and the base check on many sizes and densities;
  - rejection of malformed compact blocks (escaped gaps below 256, positions past the chunk,
    surplus escapes, class pad bits, classes or counts that disagree, reserved bits).
"""
import numpy as np
import pytest

import oracle

BASE = 0x1122334455667788


def _hand_example():
    """n = 4100 (two chunks, the second of 4 elements), old = 0x3C00 everywhere.
    chunk 0: M at 5 (x 0x03), R at 9 (x 0x8000), M at 10 (x 0x01), M at 12 (x 0x40),
             M at 300 (x 0x7F): k = 5, gaps 6 4 1 2 288 -> 288 escaped (E = 1);
             compact 5 gap bytes + 1 class byte, plus 2 bytes of X stream = 8 < version-1
             blocks 2*4 + 2*1 = 10 -> compact (the block itself is 6 bytes).
    chunk 1: M at 2 (x 0x15): k = 1, compact 1 + 1 = 2 bytes; version-1 blocks: M bitmap of
             ceil(4/8) = 1 byte (2*1 < 1 fails) + empty R list = 1 byte -> version-1 coding."""
    n = 4100
    old = np.full(n, 0x3C00, dtype=np.uint16)
    new = old.copy()
    for p, x in ((5, 0x03), (9, 0x8000), (10, 0x01), (12, 0x40), (300, 0x7F), (4096 + 2, 0x15)):
        new[p] ^= x
    expected = bytes.fromhex(
        "42463136444c5431"      # "BF16DLT1"
        "03000000" "00100000"   # version 3, 4096 elements per chunk
        "0410000000000000"      # n = 4100
        "0200000000000000"      # C = 2
        "0500000000000000"      # sum M = 5
        "0100000000000000"      # sum R = 1
        "0700000000000000"      # position bytes 6 + 1
        "6800000000000000"      # total 80 + 8 + 2 + 2 + 7 + 5 = 104
        "8877665544332211"      # base
        "0000000000000000"      # reserved
        "04020480"              # chunk 0: compact | M 4 | R 1 << 9 | E 1 << 18 = 0x80040204
        "01000000"              # chunk 1: M 1 | R 0 << 15
        "0080"                  # R stream: 0x8000
        "2001"                  # X stream: gap 288 = 0x0120
        "0604010200"            # chunk 0 gap bytes 6 4 1 2, escape
        "02"                    # chunk 0 class bits: change 1 is rare
        "04"                    # chunk 1 M bitmap: position 2 (empty R list)
        "8300f05f01"            # M stream: 0x03 0x01 0x40 0x7F 0x15, 7 bits each LSB-first
    )
    return old, new, expected


def test_hand_worked_compact_payload():
    old, new, expected = _hand_example()
    got, ck = oracle.encode(old, new, base=BASE, compact=True)
    assert got.tobytes() == expected
    st, out = oracle.decode(old, got, ck)
    assert st == oracle.OK and np.array_equal(out, new)
    st, out, ck2 = oracle.decode_incremental(old, got, oracle.checksum(old), ck)
    assert st == oracle.ERR_BASE                     # bound to BASE, not to checksum(old)
    st, out, ck2 = oracle.decode_incremental(old, got, BASE, ck)
    assert st == oracle.ERR_CHECKSUM                 # BASE is not checksum(old) either


def _pair(n, rate, seed):
    rng = np.random.default_rng(seed)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    k = int(pick.sum())
    vals = np.where(rng.random(k) < 0.97, rng.integers(1, 128, k),
                    rng.integers(1, 1 << 16, k) | 0x8000)
    new[pick] ^= vals.astype(np.uint16)
    return old, new


@pytest.mark.parametrize("n", [1, 3, 4096, 4097, 3 * 4096 + 77, 40000])
@pytest.mark.parametrize("rate", [0.0, 0.00085, 0.01, 0.02, 0.05, 0.12, 0.3, 1.0])
def test_roundtrip_and_size_bound(n, rate):
    old, new = _pair(n, rate, seed=n + int(rate * 1e5))
    base = oracle.checksum(old)
    p1, ck1 = oracle.encode(old, new)
    p3, ck3 = oracle.encode(old, new, base=base, compact=True)
    assert ck1 == ck3
    assert p3.size <= p1.size + 16
    st, out = oracle.decode(old, p3, ck3)
    assert st == oracle.OK and np.array_equal(out, new)
    st, out, ck = oracle.decode_incremental(old, p3, base, ck3)
    assert st == oracle.OK and ck == ck3
    assert oracle.decode_incremental(old, p3, base ^ 2, ck3)[0] == oracle.ERR_BASE


def test_compact_smaller_at_two_percent():
    old, new = _pair(64 * 4096, 0.02, seed=1)
    p1, _ = oracle.encode(old, new)
    p3, _ = oracle.encode(old, new, base=0, compact=True)
    assert p3.size < 0.78 * p1.size


def test_malformed_compact_blocks_rejected():
    old, new, good = _hand_example()
    good = np.frombuffer(good, dtype=np.uint8).copy()
    _, ck = oracle.encode(old, new, base=BASE, compact=True)
    x_at, gaps_at, cls_at, ct_at = 80 + 8 + 2, 80 + 8 + 2 + 2, 80 + 8 + 2 + 2 + 5, 80
    cases = {
        "escaped gap below 256": (x_at + 1, 0x01, 0x00),   # X value 288 -> 32
        "position past the chunk": (x_at + 1, 0x01, 0x10),  # X value 0x1020: 12 + 4128 >= 4096
        "more escapes than E": (gaps_at + 2, 0x01, 0x00),
        "class pad bit": (cls_at, 0x02, 0x22),
        "classes disagree with R": (cls_at, 0x02, 0x03),    # two rare, count table says one
        "entry reserved bits": (ct_at + 3, 0x80, 0x88),
        "escape count": (ct_at + 2, 0x04, 0x08),           # E = 2 with one escape byte
    }
    for name, (at, before, after) in cases.items():
        assert good[at] == before, name
        bad = good.copy()
        bad[at] = after
        assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT, name
