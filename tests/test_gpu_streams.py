"""Batched calls running concurrently on several CUDA streams (GPU).

Every call works in its own workspace and enqueues on the stream it is given, so independent
updates may run at the same time: four updates in different formats (version 1, version 3,
version 4, a version-3 overwrite payload) compressed and applied on four streams with no
synchronisation between them, and the same update compressed twice at once from the same
inputs.  Payload bytes must be the oracle's and every apply must restore new exactly.
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


def _pairs(seed, sizes, rate):
    rng = np.random.default_rng(seed)
    out = []
    for n in sizes:
        o = rng.integers(0, 1 << 16, n, dtype=np.uint16)
        nw = o.copy()
        pick = rng.random(n) < rate
        k = int(pick.sum())
        vals = np.where(rng.random(k) < 0.05, rng.integers(1, 1 << 16, k) | 0x8000,
                        rng.integers(1, 128, k))
        nw[pick] ^= vals.astype(np.uint16)
        out.append((o, nw))
    return out


KINDS = [dict(), dict(compact=True), dict(rice=True), dict(compact=True, overwrite=True)]


def test_independent_updates_on_four_streams():
    sizes = [4096 * 50 + 3, 70001, 4096 * 7, 12345]
    jobs = []
    for i, kind in enumerate(KINDS):
        pairs = _pairs(100 + i, sizes, rate=0.02 + 0.03 * i)
        olds = [from_np_u16(p[0]) for p in pairs]
        news = [from_np_u16(p[1]) for p in pairs]
        cks = [oracle.checksum(p[0]) for p in pairs]
        kw = dict(kind)
        if kind:
            kw["base_checksums"] = bd._u64_tensor(cks, "cuda")
        jobs.append(dict(pairs=pairs, olds=olds, news=news, cks=cks, kind=kind,
                         comp=bd.CompressBatch(olds, news, **kw), stream=torch.cuda.Stream()))
    torch.cuda.synchronize()
    for rnd in range(3):
        for jb in jobs:   # all compresses in flight at once
            jb["comp"].run(jb["stream"])
        for jb in jobs:
            jb["stream"].synchronize()
            assert int(jb["comp"].status.item()) == bd.OK
            jb["sizes"] = [int(v) for v in jb["comp"].sizes.tolist()]
            jb["rolls"] = [o.clone() for o in jb["olds"]]
        torch.cuda.synchronize()
        for jb in jobs:   # all applies in flight at once
            jb["dec"] = bd.DecompressBatch(jb["rolls"], jb["comp"].payloads, jb["sizes"],
                                           jb["comp"].checksums)
            jb["dec"].run(jb["stream"])
        torch.cuda.synchronize()
        for jb in jobs:
            assert int(jb["dec"].status.item()) == bd.OK
            for i, (o, nw) in enumerate(jb["pairs"]):
                if jb["kind"]:
                    ref, _ = oracle.encode(o, nw, base=jb["cks"][i], **jb["kind"])
                else:
                    ref, _ = oracle.encode(o, nw)
                got = jb["comp"].payloads[i][:jb["sizes"][i]].cpu().numpy()
                assert np.array_equal(got, ref), (jb["kind"], i)
                assert torch.equal(jb["rolls"][i].view(torch.int16),
                                   jb["news"][i].view(torch.int16)), (jb["kind"], i)


def test_same_update_compressed_twice_at_once():
    pairs = _pairs(7, [4096 * 300 + 11, 4096 * 20], rate=0.02)
    olds = [from_np_u16(p[0]) for p in pairs]
    news = [from_np_u16(p[1]) for p in pairs]
    cks = bd._u64_tensor([oracle.checksum(p[0]) for p in pairs], "cuda")
    a = bd.CompressBatch(olds, news, base_checksums=cks, rice=True)
    b = bd.CompressBatch(olds, news, base_checksums=cks, rice=True)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        a.run(sa)
        b.run(sb)
    torch.cuda.synchronize()
    assert int(a.status.item()) == bd.OK and int(b.status.item()) == bd.OK
    assert a.sizes.tolist() == b.sizes.tolist()
    assert torch.equal(a.checksums, b.checksums)
    for i, n in enumerate(int(v) for v in a.sizes.tolist()):
        assert torch.equal(a.payloads[i][:n], b.payloads[i][:n])
