"""Pins of the oracle's overwrite payloads (header flags bit 0), CPU only.

"Two forms of update payload" (NeMo-DCR page): changes may travel as absolute overwrites
instead of XOR masks, and "Retry-safe versioning": partial writes are retried through
overwrites.  An overwrite payload has the positions and classes of the XOR payload of the same
update; its R stream holds each rare element's new value and its M stream each mantissa-only
element's new mantissa, written into place by the decoder.

Pinned against:
  - a payload worked out by hand byte by byte (old mantissas nonzero, so the new-value streams
    differ from the XOR streams), and the hand-worked compact example of version 3 with the two
    edits an overwrite makes to it;
  - properties that fix the semantics: the restore from old, idempotence (applying to new gives
    new), the restore from any partly updated state, positions and classes identical to the
    XOR payload's, values an XOR payload may not hold (a zero mantissa, a rare value without
    sign or exponent bits) accepted;
  - the header rules: only flag bit 0 is defined; the base binding still holds for the
    incremental apply.
"""
import numpy as np
import pytest

import oracle

BASE = 0x1122334455667788


def _hand_v2():
    """n = 8, old = 0x3C11 everywhere; element 1 -> 0x3C14 (x = 0x0005, mantissa-only),
    element 5 -> 0xBC11 (x = 0x8000, sign flip, rare).  L = 8, bitmap bytes ceil(8/8) = 1:
    one entry is a bitmap (2*1 < 1 fails), so both blocks are 1-byte bitmaps."""
    old = np.full(8, 0x3C11, dtype=np.uint16)
    new = old.copy()
    new[1] = 0x3C14
    new[5] = 0xBC11
    header = (
        "42463136444c5431"      # "BF16DLT1"
        "02000000" "00100000"   # version 2, 4096 elements per chunk
        "0800000000000000"      # n = 8
        "0100000000000000"      # C = 1
        "0100000000000000"      # sum M = 1
        "0100000000000000"      # sum R = 1
        "0200000000000000"      # position bytes: two 1-byte bitmaps
        "5900000000000000"      # total 80 + 4 + 2 + 2 + 1 = 89
        "8877665544332211")     # base
    tail = ("0100" "0100"        # count table: M 1, R 1
            "{r}"                # R stream
            "02" "20"            # M bitmap (position 1), R bitmap (position 5)
            "{m}")               # M stream: one 7-bit value
    xor = bytes.fromhex(header + "0000000000000000" + tail.format(r="0080", m="05"))
    ovw = bytes.fromhex(header + "0100000000000000" + tail.format(r="11bc", m="14"))
    return old, new, xor, ovw


def test_hand_worked_overwrite_payload():
    old, new, xor, ovw = _hand_v2()
    got, ck = oracle.encode(old, new, base=BASE, overwrite=True)
    assert got.tobytes() == ovw
    got_x, ck_x = oracle.encode(old, new, base=BASE)
    assert got_x.tobytes() == xor and ck_x == ck
    for start in (old, new):
        st, out = oracle.decode(start, got, ck)
        assert st == oracle.OK and np.array_equal(out, new)
    # the XOR payload applied to new gives back old instead
    st, out = oracle.decode(new, got_x, ck)
    assert st == oracle.ERR_CHECKSUM and np.array_equal(out, old)


def test_hand_worked_compact_overwrite():
    """The version-3 hand example (old = 0x3C00, mantissas zero): the overwrite payload is the
    XOR payload with flags 1 and the one rare value 0x8000 replaced by the new value 0xBC00;
    the mantissa values are unchanged because old's mantissas are zero."""
    from tests.test_oracle_compact import _hand_example, BASE as B3
    old, new, expected = _hand_example()
    want = bytearray(expected)
    assert want[72] == 0 and want[88:90] == bytes.fromhex("0080")
    want[72] = 1
    want[88:90] = bytes.fromhex("00bc")
    got, ck = oracle.encode(old, new, base=B3, compact=True, overwrite=True)
    assert got.tobytes() == bytes(want)
    st, out = oracle.decode(new, got, ck)
    assert st == oracle.OK and np.array_equal(out, new)


def _pair(n, rate, seed):
    rng = np.random.default_rng(seed)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    k = int(pick.sum())
    vals = np.where(rng.random(k) < 0.9, rng.integers(1, 128, k),
                    rng.integers(1, 1 << 16, k) | 0x0080)
    new[pick] ^= vals.astype(np.uint16)
    return old, new


@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("n,rate", [(1, 1.0), (7, 0.5), (4096, 0.02), (4097, 0.3),
                                    (3 * 4096 + 77, 0.05), (20000, 0.001), (9000, 0.0)])
def test_overwrite_semantics(n, rate, compact):
    old, new = _pair(n, rate, seed=n + int(rate * 1000))
    base = oracle.checksum(old)
    ow, ck = oracle.encode(old, new, base=base, compact=compact, overwrite=True)
    xo, ck2 = oracle.encode(old, new, base=base, compact=compact)
    assert ck == ck2 == oracle.checksum(new) and ow.size == xo.size
    # identical but for the flags and the value streams
    C = (n + 4095) // 4096
    n_m = int.from_bytes(xo[32:40].tobytes(), "little")
    n_r = int.from_bytes(xo[40:48].tobytes(), "little")
    m_at = xo.size - (7 * n_m + 7) // 8
    r_at = 80 + 4 * C
    same = np.ones(xo.size, dtype=bool)
    same[72] = False
    same[r_at:r_at + 2 * n_r] = False
    same[m_at:] = False
    assert np.array_equal(ow[same], xo[same])
    assert ow[72] == 1 and xo[72] == 0
    # from old, from new, from a random mix of the two: always new
    rng = np.random.default_rng(1)
    mix = np.where(rng.random(n) < 0.5, old, new).astype(np.uint16)
    for start in (old, new, mix):
        st, out = oracle.decode(start, ow, ck)
        assert st == oracle.OK and np.array_equal(out, new)
    # incremental from old (bound to its checksum), and the base check on a partial state
    st, out, ck_inc = oracle.decode_incremental(old, ow, base, ck)
    assert st == oracle.OK and ck_inc == ck and np.array_equal(out, new)
    if not np.array_equal(mix, old):
        assert oracle.decode_incremental(mix, ow, oracle.checksum(mix), ck)[0] == oracle.ERR_BASE


def test_values_an_xor_payload_may_not_hold():
    """A mantissa-only change to mantissa 0 and a rare change to a value without sign or
    exponent bits: the XOR payload holds nonzero masks, the overwrite payload the new values
    0x00 and 0x0001, which its decoder accepts."""
    old = np.array([0x3C15, 0x3C00, 0x4000, 0x4001], dtype=np.uint16)
    new = np.array([0x3C00, 0x3C00, 0x0001, 0x4001], dtype=np.uint16)
    base = oracle.checksum(old)
    for compact in (False, True):
        ow, ck = oracle.encode(old, new, base=base, compact=compact, overwrite=True)
        st, out = oracle.decode(old, ow, ck)
        assert st == oracle.OK and np.array_equal(out, new)
        xo, _ = oracle.encode(old, new, base=base, compact=compact)
        assert oracle.decode(old, xo, ck)[0] == oracle.OK


def test_flag_rules():
    old, new, _, ovw = _hand_v2()
    ow = np.frombuffer(ovw, dtype=np.uint8).copy()
    ck = oracle.checksum(new)
    for byte, val in ((72, 3), (72, 2), (73, 1), (79, 0x80)):
        bad = ow.copy()
        bad[byte] = val
        assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT, (byte, val)
    # version 1 has no flags word: overwrite needs a bound payload
    with pytest.raises(ValueError):
        oracle.encode(old, new, overwrite=True)
