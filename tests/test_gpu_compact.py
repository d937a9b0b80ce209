"""GPU parity of version-3 payloads (compact position blocks) against the oracle.

Integer work, tolerance 0: compress in format 3 must produce the oracle's version-3 bytes at
every density -- sparse chunks that stay on version-1 lists, compact chunks that fit the
compress slot, compact chunks with more changes than a slot holds (253..508, emitted by the
dense path), and chunks too dense for a compact block.  Every decompress entry point (full,
incremental, batched, without a workspace) must restore new from them and return the
oracle's status on malformed payloads.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import from_np_u16, to_np_u16

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()


def _pair(n, rate, seed, rare=0.03):
    """Random old; new differs at a `rate` fraction of positions, a `rare` fraction of the
    changes touching sign or exponent bits."""
    rng = np.random.default_rng(seed)
    old = rng.integers(0, 1 << 16, n, dtype=np.uint16)
    new = old.copy()
    pick = rng.random(n) < rate
    k = int(pick.sum())
    vals = np.where(rng.random(k) < rare, rng.integers(1, 1 << 16, k) | 0x8000,
                    rng.integers(1, 128, k))
    new[pick] ^= vals.astype(np.uint16)
    return old, new


def _compress3(o, nw, base):
    old, new = from_np_u16(o), from_np_u16(nw)
    payload, size, ck, st = bd.compress(old, new, base_checksum=base, compact=True)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    return old, new, payload, int(size.item()), bd.u64(ck)[0]


@pytest.mark.parametrize("n", [1, 5, 4095, 4096, 4097, 3 * 4096 + 77, 40 * 4096 + 13])
@pytest.mark.parametrize("rate", [0.0, 0.00085, 0.003, 0.02, 0.05, 0.09, 0.12, 0.3, 1.0])
def test_compact_payload_bytes_and_every_apply(n, rate):
    o, nw = _pair(n, rate, seed=n * 7 + int(rate * 1e5))
    base = oracle.checksum(o)
    ref, ck_ref = oracle.encode(o, nw, base=base, compact=True)
    old, new, payload, size, ck = _compress3(o, nw, base)
    assert size == ref.size and ck == ck_ref
    assert np.array_equal(payload[:size].cpu().numpy(), ref)
    ckt = bd._u64_tensor([ck], "cuda")
    # full apply, out of place
    out = torch.empty_like(old)
    st = bd.decompress(old, payload, size, ckt, out=out)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    assert torch.equal(out.view(torch.int16), new.view(torch.int16))
    # incremental apply in place, then back
    w = old.clone()
    st, ck2 = bd.decompress_incremental(w, payload, size, base, ckt)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK and bd.u64(ck2)[0] == ck_ref
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))
    # the no-workspace entry point decodes every chunk with the block decoder
    lib = bd._lib.load()
    out2 = torch.empty_like(old)
    stn = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.bd_decompress_noalloc(old.data_ptr(), n, payload.data_ptr(), size, ckt.data_ptr(),
                                   out2.data_ptr(), stn.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == bd.OK
    torch.cuda.synchronize()
    assert int(stn.item()) == bd.OK
    assert torch.equal(out2.view(torch.int16), new.view(torch.int16))


def test_every_chunk_coding_appears():
    """The densities above cover the four codings; check it on one tensor that mixes them."""
    parts, rates = [], [0.0005, 0.02, 0.09, 0.4]
    for i, r in enumerate(rates):
        parts.append(_pair(8 * 4096, r, seed=100 + i))
    o = np.concatenate([p[0] for p in parts])
    nw = np.concatenate([p[1] for p in parts])
    base = oracle.checksum(o)
    ref, _ = oracle.encode(o, nw, base=base, compact=True)
    C = (o.size + 4095) // 4096
    table = ref[80:80 + 4 * C].view(np.uint32)
    compact = (table >> 31) == 1
    k = np.where(compact, (table & 0x1FF) + ((table >> 9) & 0x1FF), 0)
    assert (~compact).any() and (compact & (k <= 252)).any() and (compact & (k > 252)).any()
    _, _, payload, size, _ = _compress3(o, nw, base)
    assert np.array_equal(payload[:size].cpu().numpy(), ref)


def test_rare_heavy_and_far_apart_changes():
    """Rare-only chunks, single changes near the chunk end (escaped first gaps) and gaps of
    exactly 255 / 256 around the escape threshold."""
    n = 6 * 4096 + 100
    o = np.random.default_rng(3).integers(0, 1 << 16, n, dtype=np.uint16)
    nw = o.copy()
    for p in (4095, 4096 + 254, 4096 + 255, 4096 + 255 + 255, 4096 + 255 + 255 + 256,
              2 * 4096 + 4000, 3 * 4096 + 1, 3 * 4096 + 3000, 5 * 4096 + 99):
        nw[p] ^= 0x8001
    for p in range(4 * 4096, 5 * 4096, 37):
        nw[p] ^= 0x0005
    base = oracle.checksum(o)
    ref, ck_ref = oracle.encode(o, nw, base=base, compact=True)
    old, new, payload, size, ck = _compress3(o, nw, base)
    assert np.array_equal(payload[:size].cpu().numpy(), ref) and ck == ck_ref
    w = old.clone()
    st, _ = bd.decompress_incremental(w, payload, size, base, bd._u64_tensor([ck], "cuda"))
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))


def _status_all_paths(o, bad, ck, base):
    """(decompress, incremental, no-workspace) statuses of the GPU for payload `bad`."""
    old = from_np_u16(o)
    dp = torch.from_numpy(bad).cuda()
    ckt = bd._u64_tensor([ck], "cuda")
    st1 = bd.decompress(old, dp, bad.size, ckt, out=torch.empty_like(old))
    w = old.clone()
    st2, _ = bd.decompress_incremental(w, dp, bad.size, base, ckt)
    lib = bd._lib.load()
    stn = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(old)
    assert lib.bd_decompress_noalloc(old.data_ptr(), o.size, dp.data_ptr(), bad.size,
                                     ckt.data_ptr(), out.data_ptr(), stn.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream) == bd.OK
    torch.cuda.synchronize()
    return int(st1.item()), int(st2.item()), int(stn.item()), w, old


def test_malformed_compact_payloads_match_oracle():
    """Every byte of the count table, X stream and position section of a small version-3
    payload, each flipped in a few bits: all three GPU decoders return the oracle's status."""
    o, nw = _pair(3 * 4096 + 21, 0.015, seed=11, rare=0.2)
    base = oracle.checksum(o)
    ref, ck = oracle.encode(o, nw, base=base, compact=True)
    C = 4
    table = ref[80:80 + 4 * C].view(np.uint32)
    assert ((table >> 31) == 1).any()
    n_r = int.from_bytes(ref[40:48].tobytes(), "little")
    pos_bytes = int.from_bytes(ref[48:56].tobytes(), "little")
    x_at = 80 + 4 * C + 2 * n_r
    m_at = ref.size - (7 * int.from_bytes(ref[32:40].tobytes(), "little") + 7) // 8
    assert m_at - pos_bytes >= x_at
    rng = np.random.default_rng(5)
    offsets = list(range(80, 80 + 4 * C)) + list(range(x_at, m_at))
    seen = set()
    for off in offsets:
        for flip in (0x01, 0x80, int(rng.integers(1, 256))):
            bad = ref.copy()
            bad[off] ^= flip
            want = oracle.decode(o, bad, ck)[0]
            want_inc = oracle.decode_incremental(o, bad, base, ck)[0]
            got = _status_all_paths(o, bad, ck, base)
            assert got[:3] == (want, want_inc, want), (off, flip)
            seen.add(want)
    assert oracle.ERR_FORMAT in seen and oracle.ERR_CHECKSUM in seen


def test_compact_batch_and_incremental_batch():
    sizes = [5, 4096 * 10, 12345, 70001, 4096 * 3]
    rates = [0.3, 0.02, 1.0, 0.05, 0.1]
    pairs = [_pair(n, r, seed=40 + i) for i, (n, r) in enumerate(zip(sizes, rates))]
    olds = [from_np_u16(p[0]) for p in pairs]
    news = [from_np_u16(p[1]) for p in pairs]
    cks_old = [oracle.checksum(p[0]) for p in pairs]
    b3 = bd.CompressBatch(olds, news, base_checksums=bd._u64_tensor(cks_old, "cuda"),
                          compact=True)
    b3.run()
    torch.cuda.synchronize()
    assert int(b3.status.item()) == bd.OK
    s3 = [int(v) for v in b3.sizes.tolist()]
    for i, (o, nw) in enumerate(pairs):
        ref, _ = oracle.encode(o, nw, base=cks_old[i], compact=True)
        assert np.array_equal(b3.payloads[i][:s3[i]].cpu().numpy(), ref), i
    ws = [o.clone() for o in olds]
    inc = bd.IncrementalBatch(ws, b3.payloads, s3, bd._u64_tensor(cks_old, "cuda"), b3.checksums)
    inc.run()
    torch.cuda.synchronize()
    assert int(inc.status.item()) == bd.OK
    for i in range(len(sizes)):
        assert torch.equal(ws[i].view(torch.int16), news[i].view(torch.int16)), i
    outs = [torch.empty_like(o) for o in olds]
    dec = bd.DecompressBatch(olds, b3.payloads, s3, b3.checksums, outs)
    dec.run()
    torch.cuda.synchronize()
    assert int(dec.status.item()) == bd.OK
    for i in range(len(sizes)):
        assert torch.equal(outs[i].view(torch.int16), news[i].view(torch.int16)), i


def test_compact_on_bf16_workload_tensor():
    """A tensor of the dense checkpoint's shape mix and change model (2% rate)."""
    old, new = W.make_pair(W.Spec("t", (4096 * 64 + 300,), rate=0.02, tid=77), device="cuda")
    old, new = old.reshape(-1), new.reshape(-1)
    o, nw = to_np_u16(old), to_np_u16(new)
    base = oracle.checksum(o)
    ref, ck_ref = oracle.encode(o, nw, base=base, compact=True)
    ref1, _ = oracle.encode(o, nw)
    assert ref.size < 0.8 * ref1.size
    payload, size, ck, st = bd.compress(old, new, base_checksum=base, compact=True)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK and int(size.item()) == ref.size
    assert np.array_equal(payload[:ref.size].cpu().numpy(), ref)


@pytest.mark.parametrize("overwrite", [False, True])
def test_full_size_1gib_and_sweep_workloads(overwrite):
    """The 1 GiB N(0,1) tensor (about 22% changed: bitmap chunks, version-1 chunks among compact
    ones, chunks of 253..508 changes) and the 14336x4096 tensor at every rate of the sweep, in
    version 3 (XOR and overwrite): bytes identical to the oracle's, and every apply restores."""
    specs = W.dense1g() + W.sweep14336()
    for spec in specs:
        old, new = W.make_pair(spec, device="cuda")
        old, new = old.reshape(-1), new.reshape(-1)
        o, nw = to_np_u16(old), to_np_u16(new)
        base = oracle.checksum(o)
        ref, ck_ref = oracle.encode(o, nw, base=base, compact=True, overwrite=overwrite)
        payload, size, ck, st = bd.compress(old, new, base_checksum=base, compact=True,
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
