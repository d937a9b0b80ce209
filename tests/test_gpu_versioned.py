"""GPU parity of version-2 payloads (bound to a base version) against the oracle.

Integer work, tolerance 0: compress with a base checksum must produce the oracle's version-2
bytes; every decompress entry point accepts them; the incremental apply refuses a payload
whose base is not the checksum it is given (BD_ERR_BASE) and then writes nothing.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import to_np_u16

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()


def _pair(n, rate, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    old = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    return old, W.mutate(old, rate, g)


@pytest.mark.parametrize("n", [1, 7, 4095, 4096, 4097, 65536 + 3])
@pytest.mark.parametrize("rate", [0.0, 0.02, 1.0])
def test_versioned_payload_bytes_and_apply(n, rate):
    old, new = _pair(n, rate, seed=n + int(rate * 100))
    o, nw = to_np_u16(old), to_np_u16(new)
    base = oracle.checksum(o)
    ref, ck_ref = oracle.encode(o, nw, base=base)
    payload, size, ck, st = bd.compress(old, new, base_checksum=base)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    size = int(size.item())
    assert size == ref.size and bd.u64(ck)[0] == ck_ref
    assert np.array_equal(payload[:size].cpu().numpy(), ref)
    # full apply (no base check), out of place
    out = torch.empty_like(old)
    st2 = bd.decompress(old, payload, size, ck, out=out)
    torch.cuda.synchronize()
    assert int(st2.item()) == bd.OK
    assert torch.equal(out.view(torch.int16), new.view(torch.int16))
    # incremental apply with the right base
    w = old.clone()
    st3, ck3 = bd.decompress_incremental(w, payload, size, base, ck)
    torch.cuda.synchronize()
    assert int(st3.item()) == bd.OK and bd.u64(ck3)[0] == ck_ref
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))


def test_wrong_base_is_refused_and_nothing_written():
    old, new = W.make_pair(W.Spec("b", (4096 * 40 + 9,), rate=0.05, tid=31), device="cuda")
    old = old.reshape(-1)
    o = to_np_u16(old)
    base = oracle.checksum(o)
    payload, size, ck, st = bd.compress(old, new, base_checksum=base)
    size = int(size.item())
    wrong = (base + 1) & ((1 << 64) - 1)
    st_ref, _, _ = oracle.decode_incremental(o, payload[:size].cpu().numpy(), wrong, bd.u64(ck)[0])
    assert st_ref == oracle.ERR_BASE
    w = old.clone()
    st2, _ = bd.decompress_incremental(w, payload, size, wrong, ck)
    torch.cuda.synchronize()
    assert int(st2.item()) == bd.ERR_BASE
    assert torch.equal(w.view(torch.int16), old.view(torch.int16))


def test_header_corruptions_match_oracle():
    old, new = _pair(4096 * 3 + 11, 0.05, seed=5)
    o, nw = to_np_u16(old), to_np_u16(new)
    base = oracle.checksum(o)
    ref, ck = oracle.encode(o, nw, base=base)
    for off in (8, 9, 56, 64, 70, 72, 79, 80, 81):
        bad = ref.copy()
        bad[off] ^= 0x01
        for incremental in (False, True):
            if incremental:
                st_ref = oracle.decode_incremental(o, bad, base, ck)[0]
                w = old.clone()
                st, _ = bd.decompress_incremental(w, torch.from_numpy(bad).cuda(), bad.size, base, ck)
            else:
                st_ref = oracle.decode(o, bad, ck)[0]
                st = bd.decompress(old, torch.from_numpy(bad).cuda(), bad.size, ck,
                                   out=torch.empty_like(old))
            torch.cuda.synchronize()
            assert int(st.item()) == st_ref, (off, incremental)


def test_batches_mixed_versions_and_noalloc():
    sizes = [5, 4096 * 10, 12345, 70001]
    olds, news = zip(*[_pair(n, r, seed=40 + i)
                       for i, (n, r) in enumerate(zip(sizes, [0.3, 0.02, 1.0, 0.05]))])
    cks_old = [oracle.checksum(to_np_u16(o)) for o in olds]
    bases = bd._u64_tensor(cks_old, "cuda")
    b2 = bd.CompressBatch(olds, news, base_checksums=bases)
    b2.run()
    torch.cuda.synchronize()
    assert int(b2.status.item()) == bd.OK
    s2 = [int(v) for v in b2.sizes.tolist()]
    for i, (o, nw) in enumerate(zip(olds, news)):
        ref, _ = oracle.encode(to_np_u16(o), to_np_u16(nw), base=cks_old[i])
        assert np.array_equal(b2.payloads[i][:s2[i]].cpu().numpy(), ref)
    # incremental batch: tensor 2 gets a wrong base, the others apply
    ck_given = list(cks_old)
    ck_given[2] ^= 1
    ws = [o.clone() for o in olds]
    inc = bd.IncrementalBatch(ws, b2.payloads, s2, bd._u64_tensor(ck_given, "cuda"), b2.checksums)
    inc.run()
    torch.cuda.synchronize()
    st = [int(v) for v in inc.statuses.tolist()]
    assert st == [bd.OK, bd.OK, bd.ERR_BASE, bd.OK]
    assert int(inc.status.item()) == bd.ERR_BASE
    for i in range(4):
        want = olds[i] if i == 2 else news[i]
        assert torch.equal(ws[i].view(torch.int16), want.view(torch.int16)), i
    # the no-workspace entry point accepts version 2 as well
    lib = bd._lib.load()
    out = torch.empty_like(olds[1])
    stn = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = lib.bd_decompress_noalloc(olds[1].data_ptr(), olds[1].numel(), b2.payloads[1].data_ptr(),
                                   s2[1], b2.checksums.data_ptr() + 8, out.data_ptr(),
                                   stn.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == bd.OK
    torch.cuda.synchronize()
    assert int(stn.item()) == bd.OK
    assert torch.equal(out.view(torch.int16), news[1].view(torch.int16))
