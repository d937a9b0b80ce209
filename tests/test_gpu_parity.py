"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, byte for byte.

Integer work, tolerance 0: payload bytes, payload size, checksum and restored weights must be
identical to the oracle's on the same seeded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import from_np_u16, oracle_pair, to_np_u16, u64

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()
    torch.cuda.init()


def _gpu_roundtrip(old: torch.Tensor, new: torch.Tensor, inplace_check: bool = True):
    """Compresses on the GPU, checks against the oracle, applies both ways."""
    old, new = old.reshape(-1), new.reshape(-1)
    payload, size, ck, st = bd.compress(old, new)
    torch.cuda.synchronize()
    size, ck, st = int(size.item()), bd.u64(ck)[0], int(st.item())
    ref, ref_ck = oracle_pair(old, new)
    assert st == bd.OK
    assert size == ref.size, (size, ref.size)
    assert ck == ref_ck
    got = payload[:size].cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError(f"payload differs at {bad.size} bytes, first {bad[:8]}")
    # out of place
    out = torch.empty_like(old)
    s2 = bd.decompress(old, payload, size, ck, out=out)
    torch.cuda.synchronize()
    assert int(s2.item()) == bd.OK
    assert torch.equal(out.view(torch.int16), new.view(torch.int16))
    if inplace_check:
        work = old.clone()
        s3 = bd.decompress(work, payload, size, ck, out=work)
        torch.cuda.synchronize()
        assert int(s3.item()) == bd.OK
        assert torch.equal(work.view(torch.int16), new.view(torch.int16))
        # the same payload again undoes it (XOR involution), verified against checksum(old)
        ck_old = oracle.checksum(to_np_u16(old))
        s4 = bd.decompress(work, payload, size, ck_old, out=work)
        torch.cuda.synchronize()
        assert int(s4.item()) == bd.OK
        assert torch.equal(work.view(torch.int16), old.view(torch.int16))
    return payload, size, ck


def test_single_1m_parity():
    old, new = W.make_pair(W.single_1m()[0], device="cuda")
    _gpu_roundtrip(old, new)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 24, 4095, 4096, 4097, 4100, 8191, 65536 + 3,
                               3 * 4096 * 1024 + 5])
@pytest.mark.parametrize("rate", [0.0, 0.02, 0.3, 1.0])
def test_edge_sizes(n, rate):
    g = torch.Generator(device="cuda")
    g.manual_seed(n * 31 + int(rate * 1000))
    old = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    if rate < 1.0:
        new = W.mutate(old, rate, g)
    else:
        new = torch.randint(-32768, 32768, (n,), generator=g, device="cuda",
                            dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    _gpu_roundtrip(old, new)


def test_empty_tensor():
    old = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    payload, size, ck, st = bd.compress(old, old)
    torch.cuda.synchronize()
    ref, ref_ck = oracle_pair(old, old)
    assert int(size.item()) == ref.size == 64 and bd.u64(ck)[0] == ref_ck == 0
    assert np.array_equal(payload[:64].cpu().numpy(), ref)
    st = bd.decompress(old, payload, 64, 0, out=old)
    assert int(st.item()) == bd.OK


def test_exhaustive_single_bit_flips():
    i = torch.arange(1 << 20, dtype=torch.int32, device="cuda")
    old32 = i >> 4
    new32 = old32 ^ (1 << (i & 15))
    to16 = lambda v: (v - ((v >> 15) << 16)).to(torch.int16).view(torch.bfloat16)
    payload, size, ck = _gpu_roundtrip(to16(old32), to16(new32))
    assert size == 1844288


def test_bitmap_tie_and_longest_list_chunk():
    old = torch.full((4096,), 0x3F00, dtype=torch.int16, device="cuda")
    new = old.clone()
    new[0::16] ^= 0x0001
    new[1:4081:16] ^= 0x0080
    _gpu_roundtrip(old.view(torch.bfloat16), new.view(torch.bfloat16))


@pytest.mark.parametrize("spec", W.sweep14336(), ids=lambda s: s.name)
def test_sweep14336_full_size(spec):
    old, new = W.make_pair(spec, device="cuda")
    _gpu_roundtrip(old, new, inplace_check=False)


def test_dense1g_full_size():
    old, new = W.make_pair(W.dense1g()[0], device="cuda")
    _gpu_roundtrip(old, new, inplace_check=False)


def test_checksum_standalone():
    for n in [0, 1, 4, 5, 8, 20, 4097, 1 << 20, (1 << 22) + 3]:
        g = torch.Generator(device="cuda")
        g.manual_seed(n)
        w = torch.randint(-32768, 32768, (n,), generator=g, device="cuda",
                          dtype=torch.int32).to(torch.int16)
        got = bd.u64(bd.checksum(w))[0]
        assert got == oracle.checksum(to_np_u16(w)), n
    # published SplitMix64 seed-0 outputs: an all-zero tensor of 8 elements sums the first two
    z = torch.zeros(8, dtype=torch.int16, device="cuda")
    assert bd.u64(bd.checksum(z))[0] == (0xE220A8397B1DCDAF + 0x6E789E6AA1B965F4) % (1 << 64)


def test_batch_equals_single_calls():
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    sizes = [5, 4096, 0, 12345, 4096 * 1024 + 17, 1, 8192, 70000]
    olds, news = [], []
    for i, n in enumerate(sizes):
        o = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        olds.append(o)
        news.append(W.mutate(o, [0.02, 0.3, 0.0, 0.05][i % 4], g))
    b = bd.compress_batch(olds, news)
    torch.cuda.synchronize()
    assert int(b.status.item()) == bd.OK
    sizes_out = [int(v) for v in b.sizes.tolist()]
    cks = bd.u64(b.checksums)
    for i in range(len(sizes)):
        ref, ref_ck = oracle_pair(olds[i], news[i])
        assert sizes_out[i] == ref.size and cks[i] == ref_ck
        assert np.array_equal(b.payloads[i][:sizes_out[i]].cpu().numpy(), ref)
    outs = [torch.empty_like(o) for o in olds]
    d = bd.decompress_batch(olds, b.payloads, sizes_out, b.checksums, outs=outs)
    torch.cuda.synchronize()
    assert int(d.status.item()) == bd.OK
    assert all(int(s) == 0 for s in d.statuses.tolist())
    for o, nw in zip(outs, news):
        assert torch.equal(o.view(torch.int16), nw.view(torch.int16))


def test_capacity_reported():
    old, new = W.make_pair(W.single_1m()[0], device="cuda")
    old, new = old.reshape(-1), new.reshape(-1)
    ref, _ = oracle_pair(old, new)
    small = torch.empty(ref.size - 1, dtype=torch.uint8, device="cuda")
    _, size, _, st = bd.compress(old, new, payload=small)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.ERR_CAPACITY and int(size.item()) == ref.size
    exact = torch.empty(ref.size, dtype=torch.uint8, device="cuda")
    _, size, _, st = bd.compress(old, new, payload=exact)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    assert np.array_equal(exact.cpu().numpy(), ref)


def _corruptions(ref: np.ndarray):
    C = int.from_bytes(ref[24:32].tobytes(), "little")
    R = int.from_bytes(ref[40:48].tobytes(), "little")
    P = int.from_bytes(ref[48:56].tobytes(), "little")
    r_off = 64 + 4 * C
    p_off = r_off + 2 * R
    m_off = p_off + P
    out = []
    for off in (0, 9, 12, 16, 24, 32, 40, 48, 56):       # header fields
        out.append(("hdr", off, 1))
    out += [("count", 64, 1), ("count", 64 + 4 * (C - 1) + 2, 1),     # count table
            ("rare", r_off, 0xFF), ("rare", r_off + 1, 0x80),          # rare values
            ("pos", p_off, 1), ("pos", p_off + 1, 0x10), ("pos", m_off - 1, 4),
            ("mant", m_off, 1), ("mant", m_off + 3, 0x40), ("mant", ref.size - 1, 0x80)]
    return out


def test_corrupt_payload_status_matches_oracle():
    """Corruptions made on the host; GPU status (format / checksum) equals the oracle's."""
    spec = W.Spec("c", (3 * 4096 + 100,), rate=0.03)
    old, new = W.make_pair(spec, device="cuda")
    ref, ck = oracle_pair(old, new)
    o_np = to_np_u16(old)
    for kind, off, flip in _corruptions(ref):
        bad = ref.copy()
        bad[off] ^= flip
        want, _ = oracle.decode(o_np, bad, ck)
        dbad = torch.from_numpy(bad).cuda()
        out = torch.empty_like(old)
        st = bd.decompress(old, dbad, bad.size, ck, out=out)
        torch.cuda.synchronize()
        assert int(st.item()) == want, (kind, off, flip, int(st.item()), want)
    # truncated / extended payloads and a wrong element count
    for sz in (ref.size - 1, 63, 10):
        st = bd.decompress(old, torch.from_numpy(ref).cuda(), sz, ck, out=torch.empty_like(old))
        assert int(st.item()) == bd.ERR_FORMAT
    longer = np.concatenate([ref, np.zeros(16, np.uint8)])
    st = bd.decompress(old, torch.from_numpy(longer).cuda(), longer.size, ck,
                       out=torch.empty_like(old))
    assert int(st.item()) == bd.ERR_FORMAT
    st = bd.decompress(old[:-1], torch.from_numpy(ref).cuda(), ref.size, ck,
                       out=torch.empty_like(old[:-1]))
    assert int(st.item()) == bd.ERR_FORMAT
    st = bd.decompress(old, torch.from_numpy(ref).cuda(), ref.size, u64(ck ^ 1),
                       out=torch.empty_like(old))
    assert int(st.item()) == bd.ERR_CHECKSUM


def test_inplace_rollback_after_error():
    """After a failed in-place apply, applying the same payload again restores old."""
    spec = W.Spec("c", (5 * 4096,), rate=0.05)
    old, new = W.make_pair(spec, device="cuda")
    ref, ck = oracle_pair(old, new)
    for flip_at in (64 + 4 * 5 + 1, ref.size - 3):
        bad = ref.copy()
        bad[flip_at] ^= 0x21
        dbad = torch.from_numpy(bad).cuda()
        work = old.clone()
        st1 = bd.decompress(work, dbad, bad.size, ck, out=work)
        torch.cuda.synchronize()
        assert int(st1.item()) != bd.OK
        st2 = bd.decompress(work, dbad, bad.size, oracle.checksum(to_np_u16(old)), out=work)
        torch.cuda.synchronize()
        assert torch.equal(work.view(torch.int16), old.view(torch.int16))


def test_pages_api_snippet():
    """delta_compress / delta_decompress as in the API listing of the ARCv3 page."""
    g = torch.Generator(device="cuda").manual_seed(0x5EED)
    src = torch.randn(1024, 1024, dtype=torch.bfloat16, device="cuda", generator=g)
    dst = src + 1e-3 * torch.randn(src.shape, dtype=src.dtype, device="cuda", generator=g)
    compressed_diff, checksum = bd.delta_compress(src=src, dst=dst)
    restored = bd.delta_decompress(src=src, compressed_diff=compressed_diff, checksum=checksum)
    assert torch.equal(restored.view(torch.uint8), dst.view(torch.uint8))
    ref, ref_ck = oracle_pair(src, dst)
    assert checksum == ref_ck
    assert np.array_equal(compressed_diff.cpu().numpy(), ref)
    with pytest.raises(bd.DeltaError):
        bd.delta_decompress(src=src, compressed_diff=compressed_diff, checksum=checksum ^ 1)
