"""Pins of the oracle's incremental verification (CPU, no GPU).

orc_decode_incremental returns ck = ck_old + the new-minus-old checksum terms of the words the
payload changes.  Pinned against things other than itself:
  - the full checksum (whose values are pinned to the published SplitMix64 seed-0 outputs in
    test_oracle_pins.py): with ck_old = checksum(old), ck must equal checksum(new), for every
    size and change density, ragged last words included;
  - a published value directly: a 4-element tensor going from word 1 to word 0 with
    ck_old = checksum(old) must give the first SplitMix64 output for seed 0;
  - exact offsets: ck_old + d gives checksum(new) + d (mod 2^64);
  - format errors: the same status as the full decode on the same corrupt payload.
"""
import numpy as np
import pytest

import oracle

M64 = (1 << 64) - 1
SPLITMIX_SEED0_FIRST = 0xE220A8397B1DCDAF   # published SplitMix64 output 1 for seed 0


def _pair(n, rate, seed):
    rng = np.random.default_rng(seed)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    k = int(pick.sum())
    kinds = rng.random(k)
    vals = np.where(kinds < 0.97, rng.integers(1, 128, k), rng.integers(1, 1 << 16, k) | 0x8000)
    new[pick] ^= vals.astype(np.uint16)
    return old, new


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 4095, 4096, 4097, 12345])
@pytest.mark.parametrize("rate", [0.0, 0.02, 0.3, 1.0])
def test_incremental_equals_full_checksum(n, rate):
    old, new = _pair(n, rate, seed=n * 7 + int(rate * 100))
    payload, ck_new = oracle.encode(old, new)
    st, out, ck = oracle.decode_incremental(old, payload, oracle.checksum(old), ck_new)
    assert st == oracle.OK
    assert np.array_equal(out, new)
    assert ck == ck_new == oracle.checksum(new)


def test_incremental_published_value():
    old = np.array([1, 0, 0, 0], dtype=np.uint16)
    new = np.zeros(4, dtype=np.uint16)
    payload, ck_new = oracle.encode(old, new)
    assert ck_new == SPLITMIX_SEED0_FIRST
    st, _, ck = oracle.decode_incremental(old, payload, oracle.checksum(old), ck_new)
    assert st == oracle.OK and ck == SPLITMIX_SEED0_FIRST


def test_last_word_past_n_counts_as_zero():
    # the change sits in a word that straddles the end of the tensor
    for n in (5, 6, 7, 4097, 4099):
        old = np.arange(n, dtype=np.uint16) * 3 + 1
        new = old.copy()
        new[-1] ^= 0x0041
        payload, ck_new = oracle.encode(old, new)
        st, _, ck = oracle.decode_incremental(old, payload, oracle.checksum(old), ck_new)
        assert st == oracle.OK and ck == oracle.checksum(new), n


@pytest.mark.parametrize("delta", [1, 12345, M64])
def test_offset_ck_old_offsets_the_result(delta):
    old, new = _pair(9000, 0.05, seed=3)
    payload, ck_new = oracle.encode(old, new)
    ck_old = (oracle.checksum(old) + delta) & M64
    st, _, ck = oracle.decode_incremental(old, payload, ck_old, ck_new)
    assert ck == (ck_new + delta) & M64
    assert st == oracle.ERR_CHECKSUM
    st2, _, _ = oracle.decode_incremental(old, payload, ck_old, (ck_new + delta) & M64)
    assert st2 == oracle.OK


def test_no_changes_keeps_ck_old():
    old, _ = _pair(5000, 0.0, seed=9)
    payload, ck_new = oracle.encode(old, old)
    st, _, ck = oracle.decode_incremental(old, payload, 0x1234, 0x1234)
    assert st == oracle.OK and ck == 0x1234


def test_format_errors_match_full_decode():
    old, new = _pair(3 * 4096 + 17, 0.05, seed=11)
    payload, ck_new = oracle.encode(old, new)
    rng = np.random.default_rng(5)
    for at in list(rng.choice(payload.size, 40, replace=False)) + [0, 8, 16, 64, payload.size - 1]:
        bad = payload.copy()
        bad[at] ^= 0x10
        st_full, _ = oracle.decode(old, bad, ck_new)
        st_inc, _, _ = oracle.decode_incremental(old, bad, oracle.checksum(old), ck_new)
        if st_full == oracle.ERR_FORMAT:
            assert st_inc == oracle.ERR_FORMAT, at
        else:
            assert st_inc in (oracle.OK, oracle.ERR_CHECKSUM), at
