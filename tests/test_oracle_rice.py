"""Pins of the oracle's version-4 payloads (Rice-coded compact position blocks), CPU only.

Pinned against:
  - one payload worked out by hand from the version-4 layout (below, bit by bit), and every
    single-bit corruption of it rejected (format error or checksum mismatch) except in the
    base field, which a plain decode does not check;
  - a reader of the layout written here from the format definition alone (plain Python bit
    reads, no shared code with the oracle), which must restore new from old on random
    updates and agree with the oracle's chunk codings;
  - properties that follow from the encoder's choices: each compact chunk's K gives the
    fewest bits of all K in 0..7 (the smallest on a tie) and B is the bit count rounded up;
    a chunk is compact only when its block is smaller than its version-1 blocks, so the
    payload is never longer than the version-2 payload of the same update;
  - exact restore, overwrite idempotence, the incremental checksum and the base check;
  - rejection of malformed blocks (rare indices out of order or past k, a zero gap, a
    position past the chunk, a quotient running past the block, pad bits, a block longer than
    its bits, bad count entries).
"""
import numpy as np
import pytest

import oracle

BASE = 0x1122334455667788


def _hand_example():
    """n = 4100 (two chunks, the second of 4 elements), old = 0x3C00 everywhere; the update of
    the version-3 hand example.
    chunk 0: M at 5 (x 0x03), R at 9 (x 0x8000), M at 10 (x 0x01), M at 12 (x 0x40),
             M at 300 (x 0x7F): k = 5, R = 1 (index 1 of the merged list), gaps 6 4 1 2 288.
             Bits for K = 0..7: 9 + 5K + 5 + sum(g >> K) = 315 169 98 65 52 48 48 51, so
             K = 5 (tie with 6 goes to 5) and B = 6 bytes < version-1 blocks 8 + 2 = 10.
             Stream: index 1 (bits 0..8) | remainders 6 4 1 2 0 (288 mod 32) in 5 bits each
             (bits 9..33) | quotients 0 0 0 0 9 in unary (bits 34..47: 0 0 0 0 111111111 0).
             Bytes: 01 0C 09 02 C0 7F.  Entry: 1<<31 | 4 | 1<<9 | 5<<18 | 6<<21 = 0x80D40204.
    chunk 1: M at 2 (x 0x15): L = 4; Rice with k = 1: K = 1 gives 1 + 1 + 1 = 3 bits, B = 1,
             not smaller than the version-1 blocks (1-byte M bitmap + empty R list) -> plain."""
    n = 4100
    old = np.full(n, 0x3C00, dtype=np.uint16)
    new = old.copy()
    for p, x in ((5, 0x03), (9, 0x8000), (10, 0x01), (12, 0x40), (300, 0x7F), (4096 + 2, 0x15)):
        new[p] ^= x
    expected = bytes.fromhex(
        "42463136444c5431"      # "BF16DLT1"
        "04000000" "00100000"   # version 4, 4096 elements per chunk
        "0410000000000000"      # n = 4100
        "0200000000000000"      # C = 2
        "0500000000000000"      # sum M = 5
        "0100000000000000"      # sum R = 1
        "0700000000000000"      # position bytes 6 + 1
        "6600000000000000"      # total 80 + 8 + 2 + 7 + 5 = 102
        "8877665544332211"      # base
        "0000000000000000"      # flags
        "0402d480"              # chunk 0: 0x80D40204
        "01000000"              # chunk 1: M 1 | R 0 << 15
        "0080"                  # R stream: 0x8000
        "010c0902c07f"          # chunk 0 Rice block
        "04"                    # chunk 1 M bitmap: position 2 (empty R list)
        "8300f05f01"            # M stream: 0x03 0x01 0x40 0x7F 0x15, 7 bits each LSB-first
    )
    return old, new, expected


def test_hand_worked_rice_payload():
    old, new, expected = _hand_example()
    got, ck = oracle.encode(old, new, base=BASE, rice=True)
    assert got.tobytes() == expected
    st, out = oracle.decode(old, got, ck)
    assert st == oracle.OK and np.array_equal(out, new)
    st, out, ck_inc = oracle.decode_incremental(old, got, BASE, ck)
    assert st == oracle.ERR_CHECKSUM  # base matches, but BASE is not the checksum of old
    st, out, ck_inc = oracle.decode_incremental(old, got, oracle.checksum(old), ck)
    assert st == oracle.ERR_BASE      # the payload names BASE, not checksum(old)
    good, ck2 = oracle.encode(old, new, base=oracle.checksum(old), rice=True)
    st, out, ck_inc = oracle.decode_incremental(old, good, oracle.checksum(old), ck2)
    assert st == oracle.OK and ck_inc == ck2 == oracle.checksum(new)


def test_every_bit_flip_of_the_hand_payload_is_caught():
    old, new, expected = _hand_example()
    ck = oracle.checksum(new)
    ref = np.frombuffer(expected, dtype=np.uint8)
    for byte in range(ref.size):
        for bit in range(8):
            bad = ref.copy()
            bad[byte] ^= 1 << bit
            st = oracle.decode(old, bad, ck)[0]
            if 64 <= byte < 72:
                assert st == oracle.OK, (byte, bit)          # the base is not checked here
            else:
                assert st in (oracle.ERR_FORMAT, oracle.ERR_CHECKSUM), (byte, bit)


def test_hand_worked_rice_overwrite():
    """The overwrite payload of the hand example: flags 1 and the rare value replaced by the
    new value 0xBC00; old's mantissas are zero, so the mantissa values are unchanged."""
    old, new, expected = _hand_example()
    want = bytearray(expected)
    assert want[88:90] == bytes.fromhex("0080")
    want[72] = 1
    want[88:90] = bytes.fromhex("00bc")
    got, ck = oracle.encode(old, new, base=BASE, rice=True, overwrite=True)
    assert got.tobytes() == bytes(want)
    for start in (old, new):
        st, out = oracle.decode(start, got, ck)
        assert st == oracle.OK and np.array_equal(out, new)


# ---- a reader of the layout, written from the format definition --------------------------

def _bits(buf: bytes, at: int, n: int) -> int:
    return sum(((buf[(at + b) // 8] >> ((at + b) % 8)) & 1) << b for b in range(n))


def _block_len(k, L):
    bitmap = (L + 7) // 8
    return 2 * k if 2 * k < bitmap else bitmap


def _read_plain(buf, k, L):
    bitmap = (L + 7) // 8
    if 2 * k < bitmap:
        pos, p = [], 0
        for j in range(k):
            d = int.from_bytes(buf[2 * j:2 * j + 2], "little")
            p = d if j == 0 else p + d
            pos.append(p)
        return pos
    return [p for p in range(8 * bitmap) if (buf[p // 8] >> (p % 8)) & 1]


def _py_apply_v4(old: np.ndarray, payload: bytes):
    """Restores new from old and a version-4 XOR payload; returns (new, chunk codings) where a
    coding is (K, B) for a compact chunk and None for a plain one."""
    assert payload[:8] == b"BF16DLT1" and int.from_bytes(payload[8:12], "little") == 4
    n = int.from_bytes(payload[16:24], "little")
    C = int.from_bytes(payload[24:32], "little")
    n_r = int.from_bytes(payload[40:48], "little")
    pos_total = int.from_bytes(payload[48:56], "little")
    entries = [int.from_bytes(payload[80 + 4 * c:84 + 4 * c], "little") for c in range(C)]
    r_at = 80 + 4 * C
    p_at = r_at + 2 * n_r
    m_at = p_at + pos_total
    out = old.copy()
    codings = []
    mj = rj = 0
    for c, e in enumerate(entries):
        L = min(4096, n - 4096 * c)
        if e >> 31:
            km, kr, K, B = e & 0x1FF, (e >> 9) & 0x1FF, (e >> 18) & 7, (e >> 21) & 0x3FF
            blk = payload[p_at:p_at + B]
            k = km + kr
            rare_idx = {_bits(blk, 9 * j, 9) for j in range(kr)}
            u = 9 * kr + K * k
            positions, p = [], -1
            for i in range(k):
                q = 0
                while _bits(blk, u, 1):
                    q += 1
                    u += 1
                u += 1
                p += (q << K) | _bits(blk, 9 * kr + K * i, K)
                positions.append(p)
            assert (u + 7) // 8 == B
            mpos = [p for i, p in enumerate(positions) if i not in rare_idx]
            rpos = [p for i, p in enumerate(positions) if i in rare_idx]
            codings.append((K, B))
            p_at += B
        else:
            km, kr = e & 0x7FFF, (e >> 15) & 0x7FFF
            mpos = _read_plain(payload[p_at:], km, L)
            p_at += _block_len(km, L)
            rpos = _read_plain(payload[p_at:], kr, L)
            p_at += _block_len(kr, L)
            codings.append(None)
        for p in mpos:
            out[4096 * c + p] ^= _bits(payload[m_at:], 7 * mj, 7)
            mj += 1
        for p in rpos:
            out[4096 * c + p] ^= int.from_bytes(payload[r_at + 2 * rj:r_at + 2 * rj + 2], "little")
            rj += 1
    return out, codings


def _pair(n, rate, seed, rare=0.1, clustered=False):
    rng = np.random.default_rng(seed)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    if clustered:   # runs of changes: small gaps inside, long gaps between
        pick = np.repeat(rng.random((n + 15) // 16) < rate * 3, 16)[:n] & (rng.random(n) < 0.4)
    k = int(pick.sum())
    vals = np.where(rng.random(k) < rare, rng.integers(1, 1 << 16, k) | 0x0080,
                    rng.integers(1, 128, k))
    new[pick] ^= vals.astype(np.uint16)
    return old, new


def _changes(old, new, c, L):
    x = old[4096 * c:4096 * c + L] ^ new[4096 * c:4096 * c + L]
    pos = np.nonzero(x)[0]
    rare = (x[pos] & 0xFF80) != 0
    return pos, rare


@pytest.mark.parametrize("n", [1, 3, 4096, 4097, 3 * 4096 + 77, 40000])
@pytest.mark.parametrize("rate", [0.0, 0.00085, 0.01, 0.02, 0.05, 0.12, 0.3, 1.0])
def test_layout_reader_and_encoder_choices(n, rate):
    old, new = _pair(n, rate, seed=n + int(rate * 1e5))
    base = oracle.checksum(old)
    v4, ck = oracle.encode(old, new, base=base, rice=True)
    v2, _ = oracle.encode(old, new, base=base)
    assert v4.size <= v2.size
    out, codings = _py_apply_v4(old, v4.tobytes())
    assert np.array_equal(out, new)
    for c, coding in enumerate(codings):
        L = min(4096, n - 4096 * c)
        pos, rare = _changes(old, new, c, L)
        k, R = pos.size, int(rare.sum())
        plain = _block_len(k - R, L) + _block_len(R, L)
        gaps = np.diff(np.concatenate([[-1], pos]))
        cost = [9 * R + K * k + k + int((gaps >> K).sum()) for K in range(8)]
        best = int(np.argmin(cost))           # argmin takes the first, i.e. smallest, K
        fits = 1 <= k <= 508 and (cost[best] + 7) // 8 < plain
        if fits:
            assert coding == (best, (cost[best] + 7) // 8), c
        else:
            assert coding is None, c
    st, got = oracle.decode(old, v4, ck)
    assert st == oracle.OK and np.array_equal(got, new)
    st, got, ck_inc = oracle.decode_incremental(old, v4, base, ck)
    assert st == oracle.OK and ck_inc == ck and np.array_equal(got, new)
    if n > 1 and rate > 0:
        assert oracle.decode_incremental(old, v4, base ^ 1, ck)[0] == oracle.ERR_BASE


@pytest.mark.parametrize("clustered", [False, True])
def test_rice_smaller_than_byte_gaps_at_two_percent(clustered):
    old, new = _pair(64 * 4096, 0.02, seed=5, rare=0.02, clustered=clustered)
    base = oracle.checksum(old)
    v2 = oracle.encode(old, new, base=base)[0].size
    v3 = oracle.encode(old, new, base=base, compact=True)[0].size
    v4 = oracle.encode(old, new, base=base, rice=True)[0].size
    assert v4 < v3 < v2


@pytest.mark.parametrize("n,rate", [(1, 1.0), (4097, 0.3), (3 * 4096 + 77, 0.02), (9000, 0.0)])
def test_overwrite_from_any_state(n, rate):
    old, new = _pair(n, rate, seed=n)
    base = oracle.checksum(old)
    ow, ck = oracle.encode(old, new, base=base, rice=True, overwrite=True)
    xo, _ = oracle.encode(old, new, base=base, rice=True)
    assert ow.size == xo.size and ow[72] == 1 and xo[72] == 0
    mix = np.where(np.random.default_rng(3).random(n) < 0.5, old, new).astype(np.uint16)
    for start in (old, new, mix):
        st, out = oracle.decode(start, ow, ck)
        assert st == oracle.OK and np.array_equal(out, new)


def test_argument_rules():
    old, new, _ = _hand_example()
    with pytest.raises(ValueError):
        oracle.encode(old, new, rice=True)
    with pytest.raises(ValueError):
        oracle.encode(old, new, base=BASE, rice=True, compact=True)


# ---- malformed payloads -------------------------------------------------------------------

def _with_block(payload: bytes, entry: int, block: bytes, c=0) -> np.ndarray:
    """The hand payload with chunk 0's entry and Rice block replaced (sizes fixed up)."""
    p = bytearray(payload)
    old_b = (int.from_bytes(p[80:84], "little") >> 21) & 0x3FF
    blk_at = 80 + 8 + 2
    p[blk_at:blk_at + old_b] = block
    p[80:84] = entry.to_bytes(4, "little")
    pos_bytes = int.from_bytes(p[48:56], "little") - old_b + len(block)
    p[48:56] = pos_bytes.to_bytes(8, "little")
    p[56:64] = len(p).to_bytes(8, "little")
    return np.frombuffer(bytes(p), dtype=np.uint8)


def _entry(km, kr, K, B):
    return (1 << 31) | km | (kr << 9) | (K << 18) | (B << 21)


def _stream(fields):
    """Packs (value, bits) fields LSB-first and pads to whole bytes."""
    acc, at = 0, 0
    for v, nb in fields:
        acc |= v << at
        at += nb
    return acc.to_bytes((at + 7) // 8, "little"), at


def test_repacked_hand_block_is_accepted():
    """The packer below rebuilds the hand block; the malformed cases then change one thing."""
    old, new, expected = _hand_example()
    blk, used = _stream([(1, 9)] + [(g & 31, 5) for g in (6, 4, 1, 2, 288)] +
                        [(0, 1)] * 4 + [(0x1FF, 9), (0, 1)])
    assert used == 48 and blk == bytes.fromhex("010c0902c07f")
    bad = _with_block(expected, _entry(4, 1, 5, 6), blk)
    assert bad.tobytes() == expected


def _status(block_fields, entry_args, extra_bytes=b""):
    old, new, expected = _hand_example()
    blk, _ = _stream(block_fields)
    p = _with_block(expected, _entry(*entry_args), blk + extra_bytes)
    return oracle.decode(old, p, oracle.checksum(new))[0]


UNARY_OK = [(0, 1)] * 4 + [(0x1FF, 9), (0, 1)]
REM_OK = [(g & 31, 5) for g in (6, 4, 1, 2, 288)]


@pytest.mark.parametrize("case", [
    "index_past_k", "zero_gap", "quotient_past_block", "pad_bit", "block_too_long",
    "position_past_chunk", "entry_b_zero", "entry_k_zero", "entry_k_509", "k_above_chunk"])
def test_malformed_blocks_rejected(case):
    F = oracle.ERR_FORMAT
    if case == "index_past_k":
        assert _status([(5, 9)] + REM_OK + UNARY_OK, (4, 1, 5, 6)) == F
    elif case == "zero_gap":
        rem = [(0, 5)] + REM_OK[1:]              # gap 0 for the first change
        assert _status([(1, 9)] + rem + UNARY_OK, (4, 1, 5, 6)) == F
    elif case == "quotient_past_block":
        unary = [(0, 1)] * 4 + [(0x3FF, 10)]     # 48 bits, the fifth quotient unended
        assert _status([(1, 9)] + REM_OK + unary, (4, 1, 5, 6)) == F
    elif case == "pad_bit":
        # with K = 4 the block uses 9 + 20 + 5 + 18 = 52 bits: 7 bytes, 4 pad bits
        rem = [(g & 15, 4) for g in (6, 4, 1, 2, 288)]
        unary = [(0, 1)] * 4 + [((1 << 18) - 1, 18), (0, 1)]
        ok_fields = [(1, 9)] + rem + unary
        assert _status(ok_fields, (4, 1, 4, 7)) == oracle.OK
        blk, used = _stream(ok_fields)
        assert used == 52
        blk = bytearray(blk)
        blk[6] |= 0x80                           # a pad bit
        old, new, expected = _hand_example()
        p = _with_block(expected, _entry(4, 1, 4, 7), bytes(blk))
        assert oracle.decode(old, p, oracle.checksum(new))[0] == F
    elif case == "block_too_long":
        assert _status([(1, 9)] + REM_OK + UNARY_OK, (4, 1, 5, 7), b"\x00") == F
    elif case == "position_past_chunk":
        # last gap 288 + 4096: quotient 137 instead of 9 (a block of 22 bytes)
        unary = [(0, 1)] * 4 + [((1 << 137) - 1, 137), (0, 1)]
        assert _status([(1, 9)] + REM_OK + unary, (4, 1, 5, 22)) == F
    elif case == "entry_b_zero":
        assert _status([(1, 9)] + REM_OK + UNARY_OK, (4, 1, 5, 0)) == F
    elif case == "entry_k_zero":
        assert _status([(1, 9)] + REM_OK + UNARY_OK, (0, 0, 5, 6)) == F
    elif case == "entry_k_509":
        assert _status([(1, 9)] + REM_OK + UNARY_OK, (508, 1, 5, 6)) == F
    elif case == "k_above_chunk":
        # M + R = 5 on a chunk of 4 elements: chunk 1 made compact with 5 changes
        old, new, expected = _hand_example()
        p = bytearray(expected)
        p[84:88] = _entry(5, 0, 0, 1).to_bytes(4, "little")
        assert oracle.decode(old, np.frombuffer(bytes(p), np.uint8), oracle.checksum(new))[0] == F


def test_rare_indices_must_ascend():
    """Two rare changes; their indices written in descending order are rejected."""
    old = np.full(4096, 0x3C00, dtype=np.uint16)
    new = old.copy()
    for p, x in ((3, 0x8000), (7, 0x01), (20, 0x4000), (33, 0x02)):
        new[p] ^= x
    base = 7
    good, ck = oracle.encode(old, new, base=base, rice=True)
    e = int.from_bytes(good[80:84].tobytes(), "little")
    assert e >> 31 and (e >> 9) & 0x1FF == 2
    blk_at = 80 + 4 + 4
    B = (e >> 21) & 0x3FF
    blk = int.from_bytes(good[blk_at:blk_at + B].tobytes(), "little")
    assert blk & 0x1FF == 0 and (blk >> 9) & 0x1FF == 2     # indices 0 and 2
    swapped = (blk & ~((1 << 18) - 1)) | 2 | (0 << 9)
    bad = good.copy()
    bad[blk_at:blk_at + B] = np.frombuffer(swapped.to_bytes(B, "little"), np.uint8)
    assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT
    same = (blk & ~((1 << 18) - 1)) | 2 | (2 << 9)        # a repeated index
    bad[blk_at:blk_at + B] = np.frombuffer(same.to_bytes(B, "little"), np.uint8)
    assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT
