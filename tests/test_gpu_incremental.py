"""GPU parity of the incremental apply (bd_decompress_incremental) against the oracle.

Integer work, tolerance 0: status, the computed checksum ck = ck_old + the new-minus-old terms
of the changed words, and the restored weights must equal the oracle's
(oracle.decode_incremental) on the same seeded inputs; with ck_old = checksum(old) the computed
checksum must also equal the full checksum of the result.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import from_np_u16, oracle_pair, to_np_u16

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")
M64 = (1 << 64) - 1


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()


def _incr(old, payload_np, ck_old, expected):
    w = old.clone()
    payload = torch.from_numpy(payload_np).cuda()
    st, ck = bd.decompress_incremental(w, payload, payload_np.size, ck_old, expected)
    torch.cuda.synchronize()
    return int(st.item()), bd.u64(ck)[0], w


def _check(old, new):
    old, new = old.reshape(-1), new.reshape(-1)
    ref, ck_new = oracle_pair(old, new)
    o = to_np_u16(old)
    ck_old = oracle.checksum(o)
    st_ref, out_ref, ck_ref = oracle.decode_incremental(o, ref, ck_old, ck_new)
    st, ck, w = _incr(old, ref, ck_old, ck_new)
    assert st == st_ref == bd.OK
    assert ck == ck_ref == ck_new
    assert np.array_equal(to_np_u16(w), out_ref)
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))
    return ref, ck_old, ck_new


@pytest.mark.parametrize("n", [1, 5, 7, 8, 4095, 4096, 4097, 12345, 65536 + 3])
@pytest.mark.parametrize("rate", [0.0, 0.02, 0.3, 1.0])
def test_edge_sizes(n, rate):
    g = torch.Generator(device="cuda")
    g.manual_seed(n * 13 + int(rate * 1000))
    old = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    new = W.mutate(old, rate, g)
    _check(old, new)


def test_single_1m_and_undo():
    old, new = W.make_pair(W.single_1m()[0], device="cuda")
    ref, ck_old, ck_new = _check(old, new)
    # applying again from new with the checksums swapped restores old
    st, ck, w = _incr(new.reshape(-1), ref, ck_new, ck_old)
    assert st == bd.OK and ck == ck_old
    assert torch.equal(w.view(torch.int16), old.reshape(-1).view(torch.int16))


@pytest.mark.parametrize("delta", [1, 987654321, M64])
def test_wrong_ck_old_matches_oracle(delta):
    old, new = W.make_pair(W.Spec("w", (3 * 4096 + 77,), rate=0.05, tid=5), device="cuda")
    old, new = old.reshape(-1), new.reshape(-1)
    ref, ck_new = oracle_pair(old, new)
    o = to_np_u16(old)
    ck_old = (oracle.checksum(o) + delta) & M64
    st_ref, _, ck_ref = oracle.decode_incremental(o, ref, ck_old, ck_new)
    st, ck, w = _incr(old, ref, ck_old, ck_new)
    assert st == st_ref == bd.ERR_CHECKSUM
    assert ck == ck_ref == (ck_new + delta) & M64
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))


def test_corrupt_payloads_match_oracle():
    old, new = W.make_pair(W.Spec("c", (5 * 4096 + 3,), rate=0.05, tid=8), device="cuda")
    old = old.reshape(-1)
    ref, ck_new = oracle_pair(old, new)
    o = to_np_u16(old)
    ck_old = oracle.checksum(o)
    rng = np.random.default_rng(21)
    for at in sorted(set(rng.choice(ref.size, 24, replace=False).tolist()) | {64, 65, 100}):
        bad = ref.copy()
        bad[at] ^= 0x24
        st_ref, _, ck_ref = oracle.decode_incremental(o, bad, ck_old, ck_new)
        st, ck, _ = _incr(old, bad, ck_old, ck_new)
        assert st == st_ref, at
        if st_ref != bd.ERR_FORMAT:
            assert ck == ck_ref, at


def test_batch_equals_single_calls():
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    sizes = [5, 4096, 12345, 4096 * 300 + 17, 1, 70000]
    rates = [0.02, 1.0, 0.05, 0.02, 0.0, 0.3]
    olds, news, pls, szs, cko, ckn = [], [], [], [], [], []
    for n, r in zip(sizes, rates):
        o = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        nw = W.mutate(o, r, g)
        ref, ck = oracle_pair(o, nw)
        olds.append(o)
        news.append(nw)
        pls.append(torch.from_numpy(ref).cuda())
        szs.append(ref.size)
        cko.append(oracle.checksum(to_np_u16(o)))
        ckn.append(ck)
    ws = [o.clone() for o in olds]
    b = bd.IncrementalBatch(ws, pls, szs, bd._u64_tensor(cko, "cuda"), bd._u64_tensor(ckn, "cuda"))
    b.run()
    torch.cuda.synchronize()
    assert int(b.status.item()) == bd.OK
    assert all(int(s) == bd.OK for s in b.statuses.tolist())
    assert bd.u64(b.checksums) == ckn
    for w, nw in zip(ws, news):
        assert torch.equal(w.view(torch.int16), nw.view(torch.int16))


@pytest.mark.parametrize("spec", W.sweep14336()[2:4] + W.dense1g(), ids=lambda s: s.name)
def test_full_size_against_full_checksum(spec):
    old, new = W.make_pair(spec, device="cuda")
    old, new = old.reshape(-1), new.reshape(-1)
    payload, size, ck_new, st = bd.compress(old, new)
    ck_old = bd.checksum(old)
    w = old.clone()
    st2, ck = bd.decompress_incremental(w, payload, int(size.item()), ck_old, ck_new)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK and int(st2.item()) == bd.OK
    assert bd.u64(ck) == bd.u64(ck_new) == bd.u64(bd.checksum(new))
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))
