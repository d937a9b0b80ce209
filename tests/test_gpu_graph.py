"""The batched calls inside CUDA graphs (GPU).

Every call enqueues its work on the given stream without synchronising the host (the tensor
table travels as kernel parameters), so a compress and the applies that follow can be captured
once and replayed: an update loop then costs one graph launch per phase.  Replays must give the
oracle's payload bytes and restore the weights exactly, in both directions, for payloads of
versions 1, 3 and 4, with the full and with the incremental apply.
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


def _pairs():
    rng = np.random.default_rng(21)
    out = []
    for n, rate in ((4096 * 40 + 5, 0.02), (70001, 0.3), (3, 1.0), (4096 * 7, 0.001)):
        o = rng.integers(0, 1 << 16, n, dtype=np.uint16)
        nw = o.copy()
        pick = rng.random(n) < rate
        nw[pick] ^= rng.integers(1, 1 << 16, int(pick.sum()), dtype=np.uint16)
        out.append((o, nw))
    return out


def _capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


@pytest.mark.parametrize("version", [1, 3, 4])
def test_compress_and_applies_replayed_from_graphs(version):
    pairs = _pairs()
    olds = [from_np_u16(p[0]) for p in pairs]
    news = [from_np_u16(p[1]) for p in pairs]
    cks_old = [oracle.checksum(p[0]) for p in pairs]
    fmt = {1: {}, 3: dict(compact=True), 4: dict(rice=True)}[version]
    refs = [oracle.encode(o, nw, base=cks_old[i], **fmt) if fmt else oracle.encode(o, nw)
            for i, (o, nw) in enumerate(pairs)]
    ck_old_t = bd._u64_tensor(cks_old, "cuda")
    kw = dict(base_checksums=ck_old_t, **fmt) if fmt else {}
    comp = bd.CompressBatch(olds, news, **kw)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        comp.run(side)                       # warm-up outside the capture
    torch.cuda.synchronize()
    sizes = [int(v) for v in comp.sizes.tolist()]
    rolls = [o.clone() for o in olds]
    fwd = bd.DecompressBatch(rolls, comp.payloads, sizes, comp.checksums)
    bwd = bd.DecompressBatch(rolls, comp.payloads, sizes, ck_old_t)
    inc = bd.IncrementalBatch(rolls, comp.payloads, sizes, ck_old_t, comp.checksums)
    with torch.cuda.stream(side):
        fwd.run(side)
        bwd.run(side)
        inc.run(side)                        # rolls back at new
        bwd.run(side)                        # and at old again
    torch.cuda.synchronize()
    g_comp = _capture(lambda: comp.run(torch.cuda.current_stream()), side)
    g_fwd = _capture(lambda: fwd.run(torch.cuda.current_stream()), side)
    g_bwd = _capture(lambda: bwd.run(torch.cuda.current_stream()), side)
    g_inc = _capture(lambda: inc.run(torch.cuda.current_stream()), side)
    for step in range(3):
        for t in comp.payloads:
            t.fill_(0xAB)                    # stale bytes must be rewritten by the replay
        g_comp.replay()
        torch.cuda.synchronize()
        assert int(comp.status.item()) == bd.OK
        for i, (ref, ck) in enumerate(refs):
            assert sizes[i] == ref.size and bd.u64(comp.checksums)[i] == ck
            assert np.array_equal(comp.payloads[i][:ref.size].cpu().numpy(), ref)
        (g_fwd if step % 2 == 0 else g_inc).replay()
        torch.cuda.synchronize()
        done = fwd if step % 2 == 0 else inc
        assert int(done.status.item()) == bd.OK
        for r, nw in zip(rolls, news):
            assert torch.equal(r.view(torch.int16), nw.view(torch.int16))
        g_bwd.replay()
        torch.cuda.synchronize()
        assert int(bwd.status.item()) == bd.OK
        for r, o in zip(rolls, olds):
            assert torch.equal(r.view(torch.int16), o.view(torch.int16))
