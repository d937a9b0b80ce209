"""GPU parity of version-4 payloads (Rice-coded compact position blocks) against the oracle.

Integer work, tolerance 0.  Every decompress entry point (full, incremental, batched, without a
workspace) must restore new from the oracle's version-4 payloads (XOR and overwrite) at every
density, and return the oracle's status on malformed ones: every single-bit corruption of the
hand-worked payload, random corruptions of a larger one, and blocks built here to break one
rule each.  Valid blocks the encoder would never write (another K, a block of 1012 bytes) must
be accepted too, since the decoder takes any canonical coding.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import from_np_u16, to_np_u16
from tests.test_oracle_rice import (REM_OK, UNARY_OK, _entry, _hand_example, _stream,
                                    _with_block)

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()


def _pair(n, rate, seed, rare=0.03, clustered=False):
    rng = np.random.default_rng(seed)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    if clustered:
        pick = np.repeat(rng.random((n + 15) // 16) < rate * 3, 16)[:n] & (rng.random(n) < 0.4)
    k = int(pick.sum())
    vals = np.where(rng.random(k) < rare, rng.integers(1, 1 << 16, k) | 0x8000,
                    rng.integers(1, 128, k))
    new[pick] ^= vals.astype(np.uint16)
    return old, new


def _noalloc(start, payload, size, ckt):
    lib = bd._lib.load()
    out = torch.empty_like(start)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert lib.bd_decompress_noalloc(start.data_ptr(), start.numel(), payload.data_ptr(), size,
                                     ckt.data_ptr(), out.data_ptr(), st.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream) == bd.OK
    return st, out


def _statuses(o, bad, ck, base):
    """(decompress, incremental, no-workspace) statuses of the GPU for payload `bad`."""
    old = from_np_u16(o)
    dp = torch.from_numpy(np.array(bad, dtype=np.uint8)).cuda()
    ckt = bd._u64_tensor([ck], "cuda")
    st1 = bd.decompress(old, dp, bad.size, ckt, out=torch.empty_like(old))
    w = old.clone()
    st2, _ = bd.decompress_incremental(w, dp, bad.size, base, ckt)
    st3, _ = _noalloc(old, dp, bad.size, ckt)
    torch.cuda.synchronize()
    return int(st1.item()), int(st2.item()), int(st3.item())


def _expect(o, bad, ck, base):
    return (oracle.decode(o, bad, ck)[0], oracle.decode_incremental(o, bad, base, ck)[0],
            oracle.decode(o, bad, ck)[0])


@pytest.mark.parametrize("overwrite", [False, True])
@pytest.mark.parametrize("n", [1, 5, 4095, 4097, 3 * 4096 + 77, 40 * 4096 + 13])
@pytest.mark.parametrize("rate", [0.0, 0.00085, 0.003, 0.02, 0.05, 0.09, 0.12, 0.3, 1.0])
def test_rice_payloads_every_apply(n, rate, overwrite):
    o, nw = _pair(n, rate, seed=n * 5 + int(rate * 1e5), rare=0.05)
    base = oracle.checksum(o)
    ref, ck = oracle.encode(o, nw, base=base, rice=True, overwrite=overwrite)
    old, new = from_np_u16(o), from_np_u16(nw)
    payload = torch.from_numpy(ref).cuda()
    ckt = bd._u64_tensor([ck], "cuda")
    starts = [old]
    if overwrite:   # applying an overwrite payload to new, or to a mix, also gives new
        mix = np.where(np.random.default_rng(n).random(n) < 0.5, o, nw).astype(np.uint16)
        starts += [new, from_np_u16(mix)]
    for start in starts:
        out = torch.empty_like(start)
        st1 = bd.decompress(start, payload, ref.size, ckt, out=out)
        st3, out3 = _noalloc(start, payload, ref.size, ckt)
        torch.cuda.synchronize()
        assert int(st1.item()) == bd.OK and int(st3.item()) == bd.OK
        assert torch.equal(out.view(torch.int16), new.view(torch.int16))
        assert torch.equal(out3.view(torch.int16), new.view(torch.int16))
    w = old.clone()
    st2, ck2 = bd.decompress_incremental(w, payload, ref.size, base, ckt)
    torch.cuda.synchronize()
    assert int(st2.item()) == bd.OK and bd.u64(ck2)[0] == ck
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))


def test_every_bit_flip_of_the_hand_payload_matches_oracle():
    old, new, expected = _hand_example()
    ck = oracle.checksum(new)
    base = 0x1122334455667788
    ref = np.frombuffer(expected, dtype=np.uint8)
    seen = set()
    for byte in range(ref.size):
        for bit in range(8):
            bad = ref.copy()
            bad[byte] ^= 1 << bit
            want = _expect(old, bad, ck, base)
            assert _statuses(old, bad, ck, base) == want, (byte, bit)
            seen.add(want[0])
    assert {oracle.OK, oracle.ERR_FORMAT, oracle.ERR_CHECKSUM} <= seen


def test_random_corruptions_match_oracle():
    """Bytes of the count table and position section of a 4-chunk payload with compact and
    plain chunks and 20% rare changes, each flipped in a few bits."""
    o, nw = _pair(3 * 4096 + 21, 0.015, seed=11, rare=0.2)
    base = oracle.checksum(o)
    ref, ck = oracle.encode(o, nw, base=base, rice=True)
    C = 4
    table = ref[80:80 + 4 * C].view(np.uint32)
    assert ((table >> 31) == 1).any()
    n_r = int.from_bytes(ref[40:48].tobytes(), "little")
    p_at = 80 + 4 * C + 2 * n_r
    m_at = ref.size - (7 * int.from_bytes(ref[32:40].tobytes(), "little") + 7) // 8
    rng = np.random.default_rng(6)
    seen = set()
    for off in list(range(80, 80 + 4 * C)) + list(range(p_at, m_at)):
        for flip in (0x01, 0x80, int(rng.integers(1, 256))):
            bad = ref.copy()
            bad[off] ^= flip
            want = _expect(o, bad, ck, base)
            assert _statuses(o, bad, ck, base) == want, (off, flip)
            seen.add(want[0])
    assert oracle.ERR_FORMAT in seen and oracle.ERR_CHECKSUM in seen


def _hand_with(fields, entry_args, extra=b""):
    old, new, expected = _hand_example()
    blk, _ = _stream(fields)
    return old, new, _with_block(expected, _entry(*entry_args), blk + extra)


@pytest.mark.parametrize("case", [
    "index_past_k", "zero_gap", "quotient_past_block", "block_too_long", "position_past_chunk",
    "entry_b_zero", "entry_k_zero", "entry_k_509", "other_k_valid", "fixed_fields_fill_block"])
def test_built_blocks_match_oracle(case):
    base = 0x1122334455667788
    if case == "index_past_k":
        old, new, p = _hand_with([(5, 9)] + REM_OK + UNARY_OK, (4, 1, 5, 6))
    elif case == "zero_gap":
        old, new, p = _hand_with([(1, 9), (0, 5)] + REM_OK[1:] + UNARY_OK, (4, 1, 5, 6))
    elif case == "quotient_past_block":
        old, new, p = _hand_with([(1, 9)] + REM_OK + [(0, 1)] * 4 + [(0x3FF, 10)], (4, 1, 5, 6))
    elif case == "block_too_long":
        old, new, p = _hand_with([(1, 9)] + REM_OK + UNARY_OK, (4, 1, 5, 7), b"\x00")
    elif case == "position_past_chunk":
        old, new, p = _hand_with([(1, 9)] + REM_OK + [(0, 1)] * 4 + [((1 << 137) - 1, 137),
                                                                    (0, 1)], (4, 1, 5, 22))
    elif case == "entry_b_zero":
        old, new, p = _hand_with([(1, 9)] + REM_OK + UNARY_OK, (4, 1, 5, 0))
    elif case == "entry_k_zero":
        old, new, p = _hand_with([(1, 9)] + REM_OK + UNARY_OK, (0, 0, 5, 6))
    elif case == "entry_k_509":
        old, new, p = _hand_with([(1, 9)] + REM_OK + UNARY_OK, (508, 1, 5, 6))
    elif case == "other_k_valid":
        # K = 4 (the encoder takes 5): 52 bits, 7 bytes, a valid coding of the same list
        rem = [(g & 15, 4) for g in (6, 4, 1, 2, 288)]
        old, new, p = _hand_with([(1, 9)] + rem + [(0, 1)] * 4 + [((1 << 18) - 1, 18), (0, 1)],
                                 (4, 1, 4, 7))
    elif case == "fixed_fields_fill_block":
        # a 4-byte block: the index and the remainders alone need 34 bits
        old, new, expected = _hand_example()
        blk, _ = _stream([(1, 9)] + REM_OK)
        p = _with_block(expected, _entry(4, 1, 5, 4), blk[:4])
    ck = oracle.checksum(new)
    want = _expect(old, p, ck, base)
    if case == "other_k_valid":
        assert want[0] == oracle.OK
    else:
        assert want[0] == oracle.ERR_FORMAT
    assert _statuses(old, p, ck, base) == want


def _one_chunk_payload(old, pos, rare, xs, K, base):
    """A version-4 payload of one full chunk coded compactly with parameter K (which need not
    be the encoder's choice): pos ascending, rare[i] the class of change i, xs[i] its XOR."""
    k, R = len(pos), int(sum(rare))
    fields = [(i, 9) for i in range(k) if rare[i]]
    gaps = np.diff(np.concatenate([[-1], pos]))
    fields += [(int(g) & ((1 << K) - 1), K) for g in gaps]
    for g in gaps:
        q = int(g) >> K
        fields += [((1 << q) - 1, q), (0, 1)]
    blk, _ = _stream(fields)
    m_vals = [x for x, r in zip(xs, rare) if not r]
    r_vals = [x for x, r in zip(xs, rare) if r]
    mbits, _ = _stream([(v, 7) for v in m_vals])
    head = (b"BF16DLT1" + (4).to_bytes(4, "little") + (4096).to_bytes(4, "little") +
            (4096).to_bytes(8, "little") + (1).to_bytes(8, "little") +
            len(m_vals).to_bytes(8, "little") + R.to_bytes(8, "little") +
            len(blk).to_bytes(8, "little"))
    body = (_entry(k - R, R, K, len(blk)).to_bytes(4, "little") +
            b"".join(v.to_bytes(2, "little") for v in r_vals) + blk + mbits)
    total = len(head) + 8 + 16 + len(body)
    p = head + total.to_bytes(8, "little") + base.to_bytes(8, "little") + bytes(8) + body
    new = old.copy()
    for q, x in zip(pos, xs):
        new[q] ^= x
    return new, np.frombuffer(p, dtype=np.uint8)


def test_valid_long_blocks_with_other_parameters():
    """Blocks far longer than the encoder writes: K = 0 with 400 rare changes spread over the
    chunk (1012 bytes, the last position 4095), and K = 7 with 508 changes; both valid."""
    rng = np.random.default_rng(8)
    old = rng.integers(0, 1 << 16, 4096, dtype=np.uint16)
    cases = []
    pos = np.sort(rng.choice(4095, 399, replace=False)).tolist() + [4095]
    xs = [int(v) | 0x4000 for v in rng.integers(1, 1 << 16, 400)]
    cases.append((pos, [1] * 400, xs, 0))
    pos = np.sort(rng.choice(4096, 508, replace=False)).tolist()
    rare = (rng.random(508) < 0.1).astype(int).tolist()
    xs = [int(rng.integers(1, 1 << 16)) | 0x0100 if r else int(rng.integers(1, 128))
          for r in rare]
    cases.append((pos, rare, xs, 7))
    base = oracle.checksum(old)
    for pos, rare, xs, K in cases:
        new, p = _one_chunk_payload(old, pos, rare, xs, K, base)
        B = (int.from_bytes(p[80:84].tobytes(), "little") >> 21) & 0x3FF
        if K == 0:
            assert B == 1012
        ck = oracle.checksum(new)
        st, out = oracle.decode(old, p, ck)
        assert st == oracle.OK and np.array_equal(out, new)
        assert _statuses(old, p, ck, base) == (oracle.OK, oracle.OK, oracle.OK)
        assert _statuses(old, p, ck, base ^ 1)[1] == oracle.ERR_BASE
        # the block with its last byte's top bit flipped (a pad bit, or a quotient's bit)
        bad = p.copy()
        bad[80 + 4 + 2 * sum(rare) + B - 1] ^= 0x80
        assert _statuses(old, bad, ck, base) == _expect(old, bad, ck, base)


def test_batches_mixing_all_versions():
    sizes = [5, 4096 * 10, 12345, 70001, 4096 * 3]
    rates = [0.3, 0.02, 1.0, 0.05, 0.01]
    pairs = [_pair(n, r, seed=70 + i) for i, (n, r) in enumerate(zip(sizes, rates))]
    bases = [oracle.checksum(p[0]) for p in pairs]
    kinds = [dict(), dict(base=bases[1], rice=True), dict(base=bases[2], compact=True),
             dict(base=bases[3], rice=True, overwrite=True), dict(base=bases[4], rice=True)]
    refs = [oracle.encode(o, nw, **kw) for (o, nw), kw in zip(pairs, kinds)]
    payloads = [torch.from_numpy(r).cuda() for r, _ in refs]
    szs = [r.size for r, _ in refs]
    cks = bd._u64_tensor([c for _, c in refs], "cuda")
    olds = [from_np_u16(p[0]) for p in pairs]
    news = [from_np_u16(p[1]) for p in pairs]
    outs = [torch.empty_like(o) for o in olds]
    dec = bd.DecompressBatch(olds, payloads, szs, cks, outs)
    dec.run()
    torch.cuda.synchronize()
    assert int(dec.status.item()) == bd.OK
    ws = [o.clone() for o in olds]
    inc = bd.IncrementalBatch(ws, payloads, szs, bd._u64_tensor(bases, "cuda"), cks)
    inc.run()
    torch.cuda.synchronize()
    assert int(inc.status.item()) == bd.OK
    for i in range(len(sizes)):
        assert torch.equal(outs[i].view(torch.int16), news[i].view(torch.int16)), i
        assert torch.equal(ws[i].view(torch.int16), news[i].view(torch.int16)), i


@pytest.mark.parametrize("clustered", [False, True])
def test_rice_on_bf16_workload_tensor(clustered):
    """A tensor of the dense checkpoint's change model at 2%, and a clustered variant."""
    if clustered:
        o, nw = _pair(4096 * 64 + 300, 0.02, seed=78, clustered=True)
    else:
        old, new = W.make_pair(W.Spec("t", (4096 * 64 + 300,), rate=0.02, tid=77),
                               device="cuda")
        o, nw = to_np_u16(old.reshape(-1)), to_np_u16(new.reshape(-1))
    base = oracle.checksum(o)
    ref, ck = oracle.encode(o, nw, base=base, rice=True)
    ref3, _ = oracle.encode(o, nw, base=base, compact=True)
    assert ref.size < ref3.size
    got = _statuses(o, ref, ck, base)
    assert got == (oracle.OK, oracle.OK, oracle.OK)


# ---- compress (format 4) -------------------------------------------------------------------

def _compress4(o, nw, base, overwrite=False):
    old, new = from_np_u16(o), from_np_u16(nw)
    payload, size, ck, st = bd.compress(old, new, base_checksum=base, rice=True,
                                        overwrite=overwrite)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    return old, new, payload, int(size.item()), bd.u64(ck)[0]


@pytest.mark.parametrize("overwrite", [False, True])
@pytest.mark.parametrize("n", [1, 5, 4095, 4096, 4097, 3 * 4096 + 77, 40 * 4096 + 13])
@pytest.mark.parametrize("rate", [0.0, 0.00085, 0.003, 0.02, 0.05, 0.09, 0.12, 0.3, 1.0])
def test_compress_writes_the_oracle_bytes(n, rate, overwrite):
    o, nw = _pair(n, rate, seed=n * 11 + int(rate * 1e5), rare=0.05)
    base = oracle.checksum(o)
    ref, ck_ref = oracle.encode(o, nw, base=base, rice=True, overwrite=overwrite)
    old, new, payload, size, ck = _compress4(o, nw, base, overwrite)
    assert size == ref.size and ck == ck_ref
    assert np.array_equal(payload[:size].cpu().numpy(), ref)
    w = old.clone()
    st, ck2 = bd.decompress_incremental(w, payload, size, base, bd._u64_tensor([ck], "cuda"))
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK and bd.u64(ck2)[0] == ck_ref
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))


def test_every_chunk_coding_appears():
    """Chunks that stay plain, compact chunks within a compress slot (<= 252 changes), compact
    chunks beyond it (253..508, emitted by the dense path) and chunks too dense for a block."""
    parts, rates = [], [0.0005, 0.02, 0.09, 0.4]
    for i, r in enumerate(rates):
        parts.append(_pair(8 * 4096, r, seed=200 + i))
    o = np.concatenate([p[0] for p in parts])
    nw = np.concatenate([p[1] for p in parts])
    base = oracle.checksum(o)
    for overwrite in (False, True):
        ref, _ = oracle.encode(o, nw, base=base, rice=True, overwrite=overwrite)
        C = (o.size + 4095) // 4096
        table = ref[80:80 + 4 * C].view(np.uint32)
        compact = (table >> 31) == 1
        k = np.where(compact, (table & 0x1FF) + ((table >> 9) & 0x1FF), 0)
        assert (~compact).any() and (compact & (k <= 252)).any() and (compact & (k > 252)).any()
        _, _, payload, size, _ = _compress4(o, nw, base, overwrite)
        assert np.array_equal(payload[:size].cpu().numpy(), ref)


def test_gap_extremes():
    """Single changes at the chunk's end (first gap 4096), gaps at powers of two around every
    K, a chunk of exactly 508 changes and one of 509, rare-only and mantissa-only chunks."""
    n = 10 * 4096 + 100
    rng = np.random.default_rng(31)
    o = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    nw = o.copy()
    nw[4095] ^= 0x0001
    p = 4096
    for g in (1, 2, 3, 4, 7, 8, 15, 16, 31, 32, 63, 64, 127, 128, 255, 256, 511, 512, 1023):
        p += g
        nw[p] ^= 0x8001 if g % 3 == 0 else 0x0011
    for c, k in ((2, 508), (3, 509)):
        pos = np.sort(rng.choice(4096, k, replace=False)) + c * 4096
        nw[pos] ^= 0x0003
    nw[4 * 4096:5 * 4096:97] ^= 0x8000                     # rare only
    nw[5 * 4096 + 1:6 * 4096:53] ^= 0x0040                 # mantissa only
    nw[6 * 4096 + 5:6 * 4096 + 300] ^= 0x0002              # a run of 295
    nw[9 * 4096 + 7] ^= 0x0100                             # tail chunk of 4096 too
    nw[n - 1] ^= 0x0005                                    # and the ragged last chunk
    base = oracle.checksum(o)
    for overwrite in (False, True):
        ref, ck_ref = oracle.encode(o, nw, base=base, rice=True, overwrite=overwrite)
        old, new, payload, size, ck = _compress4(o, nw, base, overwrite)
        assert size == ref.size and ck == ck_ref
        assert np.array_equal(payload[:size].cpu().numpy(), ref)
        out = torch.empty_like(old)
        st = bd.decompress(old, payload, size, bd._u64_tensor([ck], "cuda"), out=out)
        torch.cuda.synchronize()
        assert int(st.item()) == bd.OK
        assert torch.equal(out.view(torch.int16), new.view(torch.int16))


def test_rice_compress_batch():
    sizes = [5, 4096 * 10, 12345, 70001, 4096 * 3]
    rates = [0.3, 0.02, 1.0, 0.05, 0.1]
    pairs = [_pair(n, r, seed=240 + i) for i, (n, r) in enumerate(zip(sizes, rates))]
    olds = [from_np_u16(p[0]) for p in pairs]
    news = [from_np_u16(p[1]) for p in pairs]
    cks_old = [oracle.checksum(p[0]) for p in pairs]
    for overwrite in (False, True):
        b4 = bd.CompressBatch(olds, news, base_checksums=bd._u64_tensor(cks_old, "cuda"),
                              rice=True, overwrite=overwrite)
        b4.run()
        torch.cuda.synchronize()
        assert int(b4.status.item()) == bd.OK
        s4 = [int(v) for v in b4.sizes.tolist()]
        for i, (o, nw) in enumerate(pairs):
            ref, _ = oracle.encode(o, nw, base=cks_old[i], rice=True, overwrite=overwrite)
            assert np.array_equal(b4.payloads[i][:s4[i]].cpu().numpy(), ref), i
        ws = [o.clone() for o in olds]
        inc = bd.IncrementalBatch(ws, b4.payloads, s4, bd._u64_tensor(cks_old, "cuda"),
                                  b4.checksums)
        inc.run()
        torch.cuda.synchronize()
        assert int(inc.status.item()) == bd.OK
        for i in range(len(sizes)):
            assert torch.equal(ws[i].view(torch.int16), news[i].view(torch.int16)), i


def test_compress_on_bf16_workload_tensor():
    old, new = W.make_pair(W.Spec("t", (4096 * 64 + 300,), rate=0.02, tid=79), device="cuda")
    old, new = old.reshape(-1), new.reshape(-1)
    o, nw = to_np_u16(old), to_np_u16(new)
    base = oracle.checksum(o)
    ref, ck_ref = oracle.encode(o, nw, base=base, rice=True)
    payload, size, ck, st = bd.compress(old, new, base_checksum=base, rice=True)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK and int(size.item()) == ref.size
    assert np.array_equal(payload[:ref.size].cpu().numpy(), ref)


@pytest.mark.parametrize("overwrite", [False, True])
def test_full_size_1gib_and_sweep_workloads(overwrite):
    """The 1 GiB N(0,1) tensor (about 22% changed) and the 14336x4096 tensor at every rate of
    the sweep, in version 4: bytes identical to the oracle's, and every apply restores."""
    for spec in W.dense1g() + W.sweep14336():
        old, new = W.make_pair(spec, device="cuda")
        old, new = old.reshape(-1), new.reshape(-1)
        o, nw = to_np_u16(old), to_np_u16(new)
        base = oracle.checksum(o)
        ref, ck_ref = oracle.encode(o, nw, base=base, rice=True, overwrite=overwrite)
        payload, size, ck, st = bd.compress(old, new, base_checksum=base, rice=True,
                                            overwrite=overwrite)
        torch.cuda.synchronize()
        assert int(st.item()) == bd.OK, spec.name
        size = int(size.item())
        assert size == ref.size and bd.u64(ck)[0] == ck_ref, spec.name
        assert np.array_equal(payload[:size].cpu().numpy(), ref), spec.name
        w = old.clone()
        st2 = bd.decompress(w, payload, size, ck, out=w)
        w2 = old.clone()
        st3, ck3 = bd.decompress_incremental(w2, payload, size, base, ck)
        torch.cuda.synchronize()
        assert int(st2.item()) == bd.OK and int(st3.item()) == bd.OK, spec.name
        assert bd.u64(ck3)[0] == ck_ref, spec.name
        assert torch.equal(w.view(torch.int16), new.view(torch.int16)), spec.name
        assert torch.equal(w2.view(torch.int16), new.view(torch.int16)), spec.name
        del old, new, w, w2, payload


@pytest.mark.parametrize("kind", [dict(), dict(compact=True), dict(rice=True),
                                  dict(overwrite=True), dict(compact=True, overwrite=True),
                                  dict(rice=True, overwrite=True)])
def test_empty_tensor_in_every_bound_format(kind):
    """n = 0: the 80-byte header alone (C = 0, checksum 0) in versions 2 to 4, applied in full
    and incrementally."""
    o = np.zeros(0, dtype=np.uint16)
    base = oracle.checksum(o)   # 0
    assert oracle.decode_incremental(o, oracle.encode(o, o, base=base, **kind)[0], base, 0)[0] \
        == oracle.OK
    ref, ck_ref = oracle.encode(o, o, base=base, **kind)
    assert ref.size == 80 and ck_ref == 0
    old = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    payload, size, ck, st = bd.compress(old, old, base_checksum=base, **kind)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK and int(size.item()) == 80 and bd.u64(ck)[0] == 0
    assert np.array_equal(payload[:80].cpu().numpy(), ref)
    st1 = bd.decompress(old, payload, 80, 0, out=old)
    st2, ck2 = bd.decompress_incremental(old, payload, 80, base, bd._u64_tensor([0], "cuda"))
    torch.cuda.synchronize()
    assert int(st1.item()) == bd.OK and int(st2.item()) == bd.OK and bd.u64(ck2)[0] == 0
