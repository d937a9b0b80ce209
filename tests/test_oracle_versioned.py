"""Pins of the oracle's version-2 payloads (bound to a base version), CPU only.

Version 2 is version 1 with an 80-byte header: the version field reads 2, the total size
grows by 16, and after the 64 version-1 header bytes come the u64 base checksum and u64 zero;
every section after the header is byte-identical.  Pinned against:
  - the hand-worked version-1 payloads (tests/golden/hand_examples.json) with that header rule
    applied by hand in the test (no expected value from running code);
  - random inputs: the sections after the header equal the version-1 payload's;
  - the check order: header and count-table format errors first, then the base, then chunks.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
BASE = 0x0123456789ABCDEF


def _examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


def _arrays(ex):
    n = ex["n"]
    old = np.full(n, int(ex["old_fill"], 16), dtype=np.uint16)
    for k, v in ex["old_set"].items():
        old[int(k)] = int(v, 16)
    new = old.copy()
    for k, v in ex["xor"].items():
        new[int(k)] ^= np.uint16(int(v, 16))
    return old, new


def _v2_of(v1: bytes, base: int) -> bytes:
    """The version-2 header rule applied by hand to a version-1 payload."""
    out = bytearray(v1[:64])
    out[8:12] = (2).to_bytes(4, "little")
    total = int.from_bytes(v1[56:64], "little") + 16
    out[56:64] = total.to_bytes(8, "little")
    out += base.to_bytes(8, "little") + bytes(8)
    return bytes(out) + v1[64:]


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_hand_worked_payloads_in_version_2(idx):
    ex = _examples()[idx]
    old, new = _arrays(ex)
    v1 = bytes.fromhex("".join(ex["payload_hex"]).replace(" ", ""))
    got, ck = oracle.encode(old, new, base=BASE)
    assert got.tobytes() == _v2_of(v1, BASE), ex["name"]
    st, out = oracle.decode(old, got, ck)
    assert st == oracle.OK and np.array_equal(out, new)


@pytest.mark.parametrize("n,rate", [(1, 1.0), (4097, 0.02), (3 * 4096 + 5, 0.3), (20000, 0.0)])
def test_sections_equal_version_1(n, rate):
    rng = np.random.default_rng(n)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    new[pick] ^= rng.integers(1, 1 << 16, int(pick.sum()), dtype=np.uint16)
    base = oracle.checksum(old)
    p1, ck1 = oracle.encode(old, new)
    p2, ck2 = oracle.encode(old, new, base=base)
    assert ck1 == ck2 and p2.size == p1.size + 16
    assert p2.tobytes() == _v2_of(p1.tobytes(), base)
    st, out, ck = oracle.decode_incremental(old, p2, base, ck2)
    assert st == oracle.OK and ck == ck2 and np.array_equal(out, new)


def test_base_mismatch_and_order_of_checks():
    rng = np.random.default_rng(4)
    old = rng.integers(0, 1 << 16, 3 * 4096, dtype=np.uint16)
    new = old.copy()
    new[::50] ^= 0x0003
    base = oracle.checksum(old)
    p2, ck = oracle.encode(old, new, base=base)
    # wrong base: refused
    assert oracle.decode_incremental(old, p2, base ^ 1, ck)[0] == oracle.ERR_BASE
    # the full decode does not check the base
    assert oracle.decode(old, p2, ck)[0] == oracle.OK
    # a header format error comes first
    bad = p2.copy()
    bad[72] = 2     # a flag bit with no meaning (bit 0 marks an overwrite payload)
    assert oracle.decode_incremental(old, bad, base ^ 1, ck)[0] == oracle.ERR_FORMAT
    assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT
    # a malformed chunk comes after the base: a zero delta after the first in chunk 0's list
    bad = p2.copy()
    first = 80 + 4 * 3 + 2 * 0          # start of the position section (no rare changes)
    assert int(bad[80]) + (int(bad[81]) << 8) == 82   # 82 mantissa-only changes in chunk 0
    bad[first + 2:first + 4] = 0
    assert oracle.decode_incremental(old, bad, base ^ 1, ck)[0] == oracle.ERR_BASE
    assert oracle.decode_incremental(old, bad, base, ck)[0] == oracle.ERR_FORMAT


def test_unknown_version_rejected():
    old = np.zeros(8, dtype=np.uint16)
    new = old.copy()
    new[3] = 1
    p2, ck = oracle.encode(old, new, base=0)
    for version in (0, 5, 255):
        bad = p2.copy()
        bad[8] = version
        assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT, version
