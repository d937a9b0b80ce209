"""bd_decompress_batch_streamed on the GPU: payloads in page-locked host memory, copied
through two device slots while the previous slot's tensors are applied.

The payloads are the oracle's (integer work, tolerance 0), laid out in host memory at
arbitrary byte offsets; the slot is made small so that a call runs several groups and both
slots are refilled.  Results must equal those of the oracle's decoder: restored tensors,
per-tensor statuses and the call's largest status -- also for a corrupted payload in a later
group and for an out-of-place call -- and applying the same payloads with the checksums of
old must restore old.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import oracle_pair, to_np_u16

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()


def _tensors(seed=23):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    ns = [4096 * 40 + 3, 0, 12345, 4096 * 2, 1, 70001, 4096 * 25, 9000, 4096 * 4 + 100,
          4096 * 30, 20000]
    rates = [0.02, 0.0, 0.3, 1.0, 0.5, 0.05, 0.02, 0.0, 0.4, 0.03, 0.1]
    olds, news = [], []
    for n, r in zip(ns, rates):
        o = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        olds.append(o)
        news.append(W.mutate(o, r, g))
    return olds, news


def _groups(sizes, slot):
    """Groups the call makes: consecutive payloads, each at a 256-byte boundary, per slot."""
    groups, used = 0, slot
    for z in sizes:
        need = (z + 255) // 256 * 256
        if used + need > slot:
            groups, used = groups + 1, 0
        used += need
    return groups


def _host_layout(refs, gap=37):
    """Host buffer holding the payloads back to back at odd offsets (not 256-aligned), or with
    gap=None at 256-byte boundaries -- the slot's own layout, so that the call copies each
    group's payloads together."""
    offs, o = [], (gap or 0)
    for r in refs:
        offs.append(o)
        o += (r.size + 255) // 256 * 256 if gap is None else r.size + gap
    return offs, o


@pytest.mark.parametrize("host_kind,gap", [("mapped", 37), ("pinned", 37), ("pinned", None)])
def test_streamed_apply_matches_oracle(host_kind, gap):
    olds, news = _tensors()
    pairs = [oracle_pair(o, nw) for o, nw in zip(olds, news)]
    refs = [p[0] for p in pairs]
    cks = [p[1] for p in pairs]
    ck_old = [oracle.checksum(to_np_u16(o)) for o in olds]
    offs, total = _host_layout(refs, gap)
    if host_kind == "mapped":
        host = bd.MappedHostBuffer(total)
        view = host.numpy()
    else:
        host = torch.empty(total, dtype=torch.uint8, pin_memory=True)
        view = host.numpy()
    for r, o in zip(refs, offs):
        view[o:o + r.size] = r
    slot = (max(r.size for r in refs) + 255) // 256 * 256 + 256
    assert _groups([r.size for r in refs], slot) >= 3   # both slots refilled
    rolls = [o.clone() for o in olds]
    expected = bd._u64_tensor(cks, "cuda")
    call = bd.StreamedDecompressBatch(rolls, host, offs, [r.size for r in refs], expected,
                                      slot_bytes=slot)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        call.run(stream)
    stream.synchronize()
    assert int(call.status.item()) == bd.OK
    assert all(int(s) == bd.OK for s in call.statuses.tolist())
    for r, o, nw, ref, ck in zip(rolls, olds, news, refs, cks):
        st, restored = oracle.decode(to_np_u16(o), ref, ck)
        assert st == oracle.OK
        assert np.array_equal(to_np_u16(r), restored)
        assert torch.equal(r.view(torch.int16), nw.view(torch.int16))
    # the same host payloads with the checksums of old bring old back
    back = bd.StreamedDecompressBatch(rolls, host, offs, [r.size for r in refs],
                                      bd._u64_tensor(ck_old, "cuda"), slot_bytes=slot)
    with torch.cuda.stream(stream):
        back.run(stream)
    stream.synchronize()
    assert int(back.status.item()) == bd.OK
    for r, o in zip(rolls, olds):
        assert torch.equal(r.view(torch.int16), o.view(torch.int16))


def test_streamed_apply_reports_a_corrupted_later_group():
    olds, news = _tensors(seed=29)
    pairs = [oracle_pair(o, nw) for o, nw in zip(olds, news)]
    refs = [p[0].copy() for p in pairs]
    cks = [p[1] for p in pairs]
    # corrupt the last tensor's payload (a later group): flip a bit of its M stream
    bad = len(refs) - 1
    refs[bad][-1] ^= 0x01
    st_ref = [oracle.decode(to_np_u16(o), r, ck)[0] for o, r, ck in zip(olds, refs, cks)]
    assert st_ref[bad] != oracle.OK and all(s == oracle.OK for s in st_ref[:bad])
    offs, total = _host_layout(refs, gap=3)
    host = bd.MappedHostBuffer(total)
    for r, o in zip(refs, offs):
        host.numpy()[o:o + r.size] = r
    slot = (max(r.size for r in refs) + 255) // 256 * 256
    assert _groups([r.size for r in refs], slot) >= 3
    outs = [torch.empty_like(o) for o in olds]
    call = bd.StreamedDecompressBatch(olds, host, offs, [r.size for r in refs],
                                      bd._u64_tensor(cks, "cuda"), slot_bytes=slot, outs=outs)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        call.run(stream)
    stream.synchronize()
    got = [int(s) for s in call.statuses.tolist()]
    assert got == [int(s) for s in st_ref]
    assert int(call.status.item()) == max(got)
    for i, (out, nw) in enumerate(zip(outs, news)):
        if i != bad:
            assert torch.equal(out.view(torch.int16), nw.view(torch.int16))
    # the same statuses as the device-payload batch on the same bytes
    dev_payloads = [torch.from_numpy(r).cuda() for r in refs]
    outs2 = [torch.empty_like(o) for o in olds]
    ref_call = bd.DecompressBatch(olds, dev_payloads, [r.size for r in refs],
                                  bd._u64_tensor(cks, "cuda"), outs=outs2)
    ref_call.run()
    torch.cuda.synchronize()
    assert [int(s) for s in ref_call.statuses.tolist()] == got
    for a, b in zip(outs, outs2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
