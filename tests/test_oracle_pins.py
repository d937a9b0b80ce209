"""Pins of the CPU oracle against what the pages and the mathematics fix.

No expected value here comes from running the oracle (or the CUDA path):
  * hand-worked payloads (tests/golden/hand_examples.json) for the section order, header,
    bit order, delta coding, bitmap coding and the ragged last chunk;
  * the published SplitMix64 seed-0 sequence for the checksum;
  * the XOR identity old ^ (old ^ new) == new ("GPU-accelerated Weight Teleportation",
    section "Delta update algebra") and bit-exact restore (the API listing of "Every byte
    counts: ARCv3 ...": restored equals dst as bytes);
  * brute-force class counts computed with numpy from the field definitions;
  * the closed-form payload size and the exhaustive single-bit-flip tensor.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
M64 = (1 << 64) - 1


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _example_arrays(ex):
    n = ex["n"]
    old = np.full(n, int(ex["old_fill"], 16), dtype=np.uint16)
    for k, v in ex["old_set"].items():
        old[int(k)] = int(v, 16)
    new = old.copy()
    for k, v in ex["xor"].items():
        new[int(k)] ^= np.uint16(int(v, 16))
    return old, new


def _hex_bytes(parts):
    return bytes.fromhex("".join(parts).replace(" ", ""))


# ---------------------------------------------------------------- hand-worked payloads

@pytest.mark.parametrize("idx", [0, 1, 2])
def test_hand_worked_payload_bytes(idx):
    ex = _golden()["examples"][idx]
    old, new = _example_arrays(ex)
    payload, _ = oracle.encode(old, new)
    assert payload.tobytes() == _hex_bytes(ex["payload_hex"]), ex["name"]
    st, restored = oracle.decode(old, payload, oracle.checksum(new))
    assert st == oracle.OK
    assert restored.tobytes() == new.tobytes()


def test_full_chunk_bitmap_tie_and_longest_list():
    """n=4096: 256 mantissa-only changes (every 16th position, XOR 0x0001) sit exactly at the
    tie 2k == 512, which selects the bitmap; 255 exponent changes (positions 1+16j, XOR
    0x0080) give 2k = 510 < 512, the longest delta list.  Expected bytes built from the
    hand-derived patterns: bitmap = (01 00) x 256; M stream = the 7-byte period
    81 40 20 10 08 04 02 repeated 32 times (value 1 at every 7th bit); delta list
    [1, 16, 16, ...]; R stream = 80 00 x 255."""
    n = 4096
    old = np.full(n, 0x3F00, dtype=np.uint16)
    new = old.copy()
    new[0::16] ^= np.uint16(0x0001)
    new[1:4081:16] ^= np.uint16(0x0080)
    assert (new[1::16] != old[1::16]).sum() == 255
    hdr = (b"BF16DLT1" + (1).to_bytes(4, "little") + (4096).to_bytes(4, "little")
           + n.to_bytes(8, "little") + (1).to_bytes(8, "little")
           + (256).to_bytes(8, "little") + (255).to_bytes(8, "little")
           + (512 + 510).to_bytes(8, "little"))
    body = ((256).to_bytes(2, "little") + (255).to_bytes(2, "little")
            + bytes([0x80, 0x00]) * 255
            + bytes([0x01, 0x00]) * 256
            + (1).to_bytes(2, "little") + (16).to_bytes(2, "little") * 254
            + bytes([0x81, 0x40, 0x20, 0x10, 0x08, 0x04, 0x02]) * 32)
    size = 64 + len(body)
    expected = hdr + size.to_bytes(8, "little") + body
    payload, _ = oracle.encode(old, new)
    assert payload.tobytes() == expected
    st, restored = oracle.decode(old, payload, oracle.checksum(new))
    assert st == oracle.OK and restored.tobytes() == new.tobytes()


# ---------------------------------------------------------------- checksum

def test_checksum_published_splitmix_values():
    for case in _golden()["checksums"]["cases"]:
        if "n_zero" in case:
            w = np.zeros(case["n_zero"], dtype=np.uint16)
        else:
            w = np.array([int(v, 16) for v in case["words"]], dtype=np.uint16)
        if "expect" in case:
            want = int(case["expect"], 16)
        else:
            want = sum(int(v, 16) for v in case["expect_sum_of"]) & M64
        assert oracle.checksum(w) == want, case


def test_checksum_is_position_keyed_and_order_free():
    rng = np.random.default_rng(1)
    w = rng.integers(0, 1 << 16, size=4 * 1000 + 3, dtype=np.uint16)
    base = oracle.checksum(w)
    # swapping two distinct 64-bit words changes it
    s = w.copy()
    s[0:4], s[400:404] = w[400:404].copy(), w[0:4].copy()
    assert not np.array_equal(s, w)
    assert oracle.checksum(s) != base
    # a single flipped bit anywhere changes it (mix64 is a bijection, so never missed)
    for i in (0, 1, 2, 3, 17, 4002):
        for b in (0, 7, 15):
            f = w.copy()
            f[i] ^= np.uint16(1 << b)
            assert oracle.checksum(f) != base
    # the wrapping sum does not depend on how the tensor is split: sum of per-segment sums
    # (segments aligned to whole words, keyed by their global word index) equals the total
    # -- checked by zeroing segments: ck(w) = ck(w with A zeroed) + ck(w with B zeroed) - ck(0)
    a = w.copy(); a[:2000] = 0
    b = w.copy(); b[2000:] = 0
    z = np.zeros_like(w)
    assert (oracle.checksum(a) + oracle.checksum(b) - oracle.checksum(z)) & M64 == base


# ---------------------------------------------------------------- counts and size

def _brute_counts(old, new):
    x = (old ^ new).astype(np.uint32)
    mant = (x != 0) & ((x & 0xFF80) == 0)
    rare = (x & 0xFF80) != 0
    C = (old.size + 4095) // 4096
    m = np.array([mant[c * 4096:(c + 1) * 4096].sum() for c in range(C)], dtype=np.int64)
    r = np.array([rare[c * 4096:(c + 1) * 4096].sum() for c in range(C)], dtype=np.int64)
    return m, r


def _closed_form(n, m, r):
    C = (n + 4095) // 4096
    pos = 0
    for c in range(C):
        L = min(4096, n - 4096 * c)
        B = (L + 7) // 8
        for k in (int(m[c]), int(r[c])):
            pos += 2 * k if 2 * k < B else B
    return 64 + 4 * C + 2 * int(r.sum()) + pos + (7 * int(m.sum()) + 7) // 8


def _parse(payload):
    p = payload.tobytes()
    hdr = {k: int.from_bytes(p[o:o + 8], "little")
           for k, o in (("n", 16), ("C", 24), ("M", 32), ("R", 40), ("pos", 48), ("size", 56))}
    C = hdr["C"]
    ct = np.frombuffer(p[64:64 + 4 * C], dtype=np.uint16).reshape(C, 2) if C else \
        np.zeros((0, 2), np.uint16)
    return hdr, ct


def _mutate(rng, old, rate):
    """Synthetic delta: rate of positions changed; 97% mantissa XOR, 2.9% exponent +-1,
    0.1% sign flip (skipping exponent moves that would reach 0 or 255)."""
    new = old.copy()
    pick = rng.random(old.size) < rate
    kind = rng.random(old.size)
    idx = np.nonzero(pick)[0]
    for i in idx:
        k = kind[i]
        if k < 0.97:
            new[i] ^= np.uint16(rng.integers(1, 128))
        elif k < 0.999:
            e = (int(old[i]) >> 7) & 0xFF
            e2 = e + (1 if rng.random() < 0.5 else -1)
            if 0 < e2 < 255:
                new[i] = np.uint16((int(old[i]) & 0x807F) | (e2 << 7))
        else:
            new[i] ^= np.uint16(0x8000)
    return new


def _bf16_normal(rng, n, std):
    f = (rng.standard_normal(n) * std).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    # round to nearest even on the upper 16 bits
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


@pytest.mark.parametrize("n", [0, 1, 7, 8, 4095, 4096, 4097, 65536 + 3])
@pytest.mark.parametrize("rate", [0.0, 0.02, 0.3, 1.0])
def test_roundtrip_counts_closed_form(n, rate):
    rng = np.random.default_rng(n * 7 + int(rate * 100))
    old = _bf16_normal(rng, n, 0.02)
    new = _mutate(rng, old, rate) if rate < 1.0 else rng.integers(0, 1 << 16, n).astype(np.uint16)
    payload, ck = oracle.encode(old, new)
    m, r = _brute_counts(old, new)
    hdr, ct = _parse(payload)
    assert hdr["n"] == n and hdr["C"] == (n + 4095) // 4096
    assert np.array_equal(ct[:, 0], m) and np.array_equal(ct[:, 1], r)
    assert hdr["M"] == m.sum() and hdr["R"] == r.sum()
    assert int(m.sum() + r.sum()) == int(((old ^ new) != 0).sum())
    assert payload.size == hdr["size"] == _closed_form(n, m, r)
    assert ck == oracle.checksum(new)
    st, restored = oracle.decode(old, payload, ck)
    assert st == oracle.OK
    assert restored.tobytes() == new.tobytes()
    # XOR identity: the mask old^new applied to old gives new, and applied again gives old
    mask = old ^ new
    assert np.array_equal(old ^ mask, new) and np.array_equal(new ^ mask, old)


def test_exhaustive_single_bit_flips():
    """old_i = i >> 4, new_i = old_i ^ (1 << (i & 15)): every single-bit flip of every 16-bit
    pattern.  Bits 0-6 are mantissa-only (7 of 16), bits 7-15 rare (9 of 16); every chunk
    has M=1792, R=2304 (both bitmaps) and the size is
    64 + 4*256 + 2*589824 + 256*1024 + 7*458752/8 = 1,844,288 bytes."""
    i = np.arange(1 << 20, dtype=np.uint32)
    old = (i >> 4).astype(np.uint16)
    new = (old ^ (1 << (i & 15))).astype(np.uint16)
    payload, ck = oracle.encode(old, new)
    hdr, ct = _parse(payload)
    assert hdr["M"] == 458752 and hdr["R"] == 589824
    assert (ct[:, 0] == 1792).all() and (ct[:, 1] == 2304).all()
    assert hdr["pos"] == 256 * 1024
    assert payload.size == 1844288
    st, restored = oracle.decode(old, payload, ck)
    assert st == oracle.OK and restored.tobytes() == new.tobytes()
    # swapping old and new gives the same counts and size (XOR is symmetric)
    payload2, _ = oracle.encode(new, old)
    hdr2, ct2 = _parse(payload2)
    assert payload2.size == payload.size and np.array_equal(ct, ct2)
    st, back = oracle.decode(new, payload2, oracle.checksum(old))
    assert st == oracle.OK and back.tobytes() == old.tobytes()


def test_tiny_brute_force():
    """Every old in a 5-pattern set and every XOR in a 6-pattern set, over 3 elements."""
    olds = [0x0000, 0x3F80, 0x8001, 0x7F7F, 0xFFFF]
    xors = [0x0000, 0x0001, 0x007F, 0x0080, 0x8000, 0xFFFF]
    for a in olds:
        for b in olds:
            for c in olds:
                old = np.array([a, b, c], dtype=np.uint16)
                for x0 in xors:
                    for x1 in xors:
                        for x2 in xors:
                            new = old ^ np.array([x0, x1, x2], dtype=np.uint16)
                            payload, ck = oracle.encode(old, new)
                            m, r = _brute_counts(old, new)
                            assert payload.size == _closed_form(3, m, r)
                            st, res = oracle.decode(old, payload, ck)
                            assert st == oracle.OK and res.tobytes() == new.tobytes()


# ---------------------------------------------------------------- corrupt payloads

def _sample_payload():
    rng = np.random.default_rng(5)
    old = _bf16_normal(rng, 9000, 0.02)
    new = _mutate(rng, old, 0.05)
    payload, ck = oracle.encode(old, new)
    return old, new, payload, ck


def test_decode_rejects_bad_headers_and_sizes():
    old, new, payload, ck = _sample_payload()
    for off in (0, 8, 12, 16, 24, 32, 40, 48, 56):
        bad = payload.copy()
        bad[off] ^= 1
        assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT, off
    assert oracle.decode(old, payload[:-1], ck)[0] == oracle.ERR_FORMAT
    assert oracle.decode(old, payload[:63], ck)[0] == oracle.ERR_FORMAT
    assert oracle.decode(old[:-1], payload, ck)[0] == oracle.ERR_FORMAT
    # count table entry changed: totals no longer match the header
    bad = payload.copy()
    bad[64] ^= 1
    assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT


def test_decode_detects_checksum_mismatch_and_stream_corruption():
    old, new, payload, ck = _sample_payload()
    assert oracle.decode(old, payload, ck ^ 1)[0] == oracle.ERR_CHECKSUM
    # flip one bit of the last mantissa byte that is not a pad bit -> a different value
    hdr, _ = _parse(payload)
    bad = payload.copy()
    bad[-2] ^= 0x10
    st = oracle.decode(old, bad, ck)[0]
    assert st in (oracle.ERR_CHECKSUM, oracle.ERR_FORMAT)
    # a rare value that loses its sign/exponent bits is not canonical
    r_off = 64 + 4 * hdr["C"]
    assert hdr["R"] > 0
    bad = payload.copy()
    bad[r_off] = 0x01
    bad[r_off + 1] = 0x00
    assert oracle.decode(old, bad, ck)[0] == oracle.ERR_FORMAT
