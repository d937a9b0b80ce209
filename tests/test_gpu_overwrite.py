"""GPU parity of overwrite payloads (header flags bit 0) against the oracle.

Integer work, tolerance 0: compress with BD_FORMAT_OVERWRITE writes the oracle's bytes in
versions 2 and 3; every decoder (full, incremental, batched, without a workspace) takes old, new
and any partly updated state to new; the incremental apply from a partly updated state, bound to
that state's checksum, skips the elements already in place and returns the checksum of the
result; malformed flags and corrupted overwrite payloads give the oracle's status.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import from_np_u16

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()


def _pair(n, rate, seed, rare=0.05):
    rng = np.random.default_rng(seed)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    k = int(pick.sum())
    vals = np.where(rng.random(k) < rare, rng.integers(1, 1 << 16, k) | 0x0080,
                    rng.integers(1, 128, k))
    new[pick] ^= vals.astype(np.uint16)
    return old, new


def _mix(old, new, seed):
    rng = np.random.default_rng(seed)
    return np.where(rng.random(old.size) < 0.5, old, new).astype(np.uint16)


def _noalloc(start, payload, size, ckt):
    lib = bd._lib.load()
    out = torch.empty_like(start)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.bd_decompress_noalloc(start.data_ptr(), start.numel(), payload.data_ptr(), size,
                                   ckt.data_ptr(), out.data_ptr(), st.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == bd.OK
    return st, out


@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("n", [1, 6, 4095, 4097, 3 * 4096 + 77, 40 * 4096 + 13])
@pytest.mark.parametrize("rate", [0.0, 0.001, 0.02, 0.09, 0.3, 1.0])
def test_overwrite_bytes_and_applies(n, rate, compact):
    o, nw = _pair(n, rate, seed=n * 3 + int(rate * 1e4) + compact)
    base = oracle.checksum(o)
    ref, ck_ref = oracle.encode(o, nw, base=base, compact=compact, overwrite=True)
    old, new = from_np_u16(o), from_np_u16(nw)
    payload, size, ck, st = bd.compress(old, new, base_checksum=base, compact=compact,
                                        overwrite=True)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    size = int(size.item())
    assert size == ref.size and bd.u64(ck)[0] == ck_ref
    assert np.array_equal(payload[:size].cpu().numpy(), ref)
    ckt = bd._u64_tensor([ck_ref], "cuda")
    mix = from_np_u16(_mix(o, nw, seed=n))
    for start in (old, new, mix):
        # full apply out of place, in place, and without a workspace
        out = torch.empty_like(start)
        st1 = bd.decompress(start, payload, size, ckt, out=out)
        w = start.clone()
        st2 = bd.decompress(w, payload, size, ckt, out=w)
        st3, out3 = _noalloc(start, payload, size, ckt)
        torch.cuda.synchronize()
        for s_, r_ in ((st1, out), (st2, w), (st3, out3)):
            assert int(s_.item()) == bd.OK
            assert torch.equal(r_.view(torch.int16), new.view(torch.int16))
    # incremental from old, bound to its checksum
    w = old.clone()
    st4, ck4 = bd.decompress_incremental(w, payload, size, base, ckt)
    torch.cuda.synchronize()
    assert int(st4.item()) == bd.OK and bd.u64(ck4)[0] == ck_ref
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))


@pytest.mark.parametrize("compact", [False, True])
def test_incremental_retry_from_partial_state(compact):
    """A payload bound to the checksum of a partly updated state: the incremental apply leaves
    the elements already in place alone and its computed checksum is that of new."""
    o, nw = _pair(5 * 4096 + 300, 0.03, seed=9)
    mix = _mix(o, nw, seed=4)
    base = oracle.checksum(mix)
    ref, ck_ref = oracle.encode(o, nw, base=base, compact=compact, overwrite=True)
    st_o, out_o, ck_o = oracle.decode_incremental(mix, ref, base, ck_ref)
    assert st_o == oracle.OK and ck_o == ck_ref and np.array_equal(out_o, nw)
    payload, size, ck, st = bd.compress(from_np_u16(o), from_np_u16(nw), base_checksum=base,
                                        compact=compact, overwrite=True)
    w = from_np_u16(mix)
    st2, ck2 = bd.decompress_incremental(w, payload, int(size.item()), base, ck)
    torch.cuda.synchronize()
    assert int(st2.item()) == bd.OK and bd.u64(ck2)[0] == ck_ref
    assert np.array_equal(w.view(torch.int16).cpu().numpy().view(np.uint16), nw)


def test_values_an_xor_payload_may_not_hold():
    o = np.array([0x3C15, 0x3C00, 0x4000, 0x4001] * 1500, dtype=np.uint16)
    nw = o.copy()
    nw[0::4] = 0x3C00     # mantissa-only change to mantissa 0
    nw[2::4] = 0x0001     # rare change to a value without sign or exponent bits
    base = oracle.checksum(o)
    for compact in (False, True):
        ref, ck = oracle.encode(o, nw, base=base, compact=compact, overwrite=True)
        payload, size, _, st = bd.compress(from_np_u16(o), from_np_u16(nw), base_checksum=base,
                                           compact=compact, overwrite=True)
        assert np.array_equal(payload[:int(size.item())].cpu().numpy(), ref)
        for start in (o, nw):
            w = from_np_u16(start)
            st2 = bd.decompress(w, payload, ref.size, ck, out=w)
            torch.cuda.synchronize()
            assert int(st2.item()) == bd.OK
            assert np.array_equal(w.view(torch.int16).cpu().numpy().view(np.uint16), nw)


def test_corruptions_match_oracle():
    """Flag bits, and bytes of the count table, position section and value streams of a small
    overwrite payload in each version: every decoder returns the oracle's status."""
    o, nw = _pair(3 * 4096 + 21, 0.02, seed=17, rare=0.2)
    base = oracle.checksum(o)
    old = from_np_u16(o)
    rng = np.random.default_rng(2)
    for compact in (False, True):
        ref, ck = oracle.encode(o, nw, base=base, compact=compact, overwrite=True)
        offsets = [72, 73, 79] + [int(x) for x in rng.integers(80, ref.size, 60)]
        for off in offsets:
            bad = ref.copy()
            bad[off] ^= 0x02 if off == 72 else int(rng.integers(1, 256))
            want = oracle.decode(o, bad, ck)[0]
            want_inc = oracle.decode_incremental(o, bad, base, ck)[0]
            dp = torch.from_numpy(bad).cuda()
            ckt = bd._u64_tensor([ck], "cuda")
            st1 = bd.decompress(old, dp, bad.size, ckt, out=torch.empty_like(old))
            w = old.clone()
            st2, _ = bd.decompress_incremental(w, dp, bad.size, base, ckt)
            st3, _ = _noalloc(old, dp, bad.size, ckt)
            torch.cuda.synchronize()
            got = (int(st1.item()), int(st2.item()), int(st3.item()))
            assert got == (want, want_inc, want), (compact, off)


def test_batches_mixing_xor_and_overwrite():
    """A decompress batch holding XOR and overwrite payloads of versions 1 to 3 together."""
    sizes = [5, 4096 * 6, 12345, 70001]
    pairs = [_pair(n, r, seed=60 + i) for i, (n, r) in enumerate(zip(sizes, [0.3, 0.02, 1.0, 0.05]))]
    olds = [from_np_u16(p[0]) for p in pairs]
    news = [from_np_u16(p[1]) for p in pairs]
    bases = [oracle.checksum(p[0]) for p in pairs]
    kinds = [dict(), dict(base_checksum=bases[1], overwrite=True),
             dict(base_checksum=bases[2], compact=True), dict(base_checksum=bases[3],
                                                            compact=True, overwrite=True)]
    payloads, szs, cks = [], [], []
    for i, kw in enumerate(kinds):
        p, s_, c_, st = bd.compress(olds[i], news[i], **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == bd.OK
        payloads.append(p)
        szs.append(int(s_.item()))
        cks.append(bd.u64(c_)[0])
    outs = [o.clone() for o in olds]
    dec = bd.DecompressBatch(outs, payloads, szs, bd._u64_tensor(cks, "cuda"))
    dec.run()
    torch.cuda.synchronize()
    assert int(dec.status.item()) == bd.OK
    for i in range(4):
        assert torch.equal(outs[i].view(torch.int16), news[i].view(torch.int16)), i
    ws = [o.clone() for o in olds]
    inc = bd.IncrementalBatch(ws, payloads, szs, bd._u64_tensor(bases, "cuda"),
                              bd._u64_tensor(cks, "cuda"))
    # item 0 is version 1 (no base): its ck_old is checksum(old) as well
    inc.run()
    torch.cuda.synchronize()
    assert int(inc.status.item()) == bd.OK
    for i in range(4):
        assert torch.equal(ws[i].view(torch.int16), news[i].view(torch.int16)), i
