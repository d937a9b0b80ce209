"""Parity at full size on the 7B-shaped dense checkpoint and the 30B-shaped MoE checkpoint, in
the launch configuration the benchmark times: one batched compress over every tensor of the
checkpoint (held in one flat buffer per checkpoint, tensors at 256-byte aligned offsets), then
one batched in-place apply on a copy of old; the dense checkpoint also in version 3 (compact
position blocks) and version 4 (Rice-coded compact position blocks).

The oracle checks a sample of tensors one by one (payload bytes, size, checksum; integer work,
tolerance 0).  Every tensor is checked by properties that hold at any size: each status is OK,
the restored checkpoint equals new bit for bit, and applying the same payloads again with the
checksums of old restores old exactly.
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


def _flat(specs, dev):
    ns = [s.numel for s in specs]
    offs, o = [], 0
    for n in ns:
        offs.append(o)
        o += (n + 127) // 128 * 128
    O = torch.empty(o, dtype=torch.bfloat16, device=dev)
    N = torch.empty(o, dtype=torch.bfloat16, device=dev)
    for s, off, n in zip(specs, offs, ns):
        a, b = W.make_pair(s, device=dev)
        O[off:off + n].copy_(a.reshape(-1))
        N[off:off + n].copy_(b.reshape(-1))
        del a, b
    return O, N, offs, ns


def _cap_estimate(spec) -> int:
    """Generous payload room for a tensor with the spec's change rate (not a bound)."""
    n = spec.numel
    C = (n + 4095) // 4096
    lam = spec.rate * 4096
    per_chunk = 1024 if lam > 100 else int(6 * lam) + 256
    return min(bd.compress_bound(n), 64 + 4 * C + per_chunk * C + int(3 * spec.rate * n) + 4096)


def _check_workload(specs, sample, compact=False, rice=False):
    dev = torch.device("cuda")
    O, N, offs, ns = _flat(specs, dev)
    olds = [O[off:off + n] for off, n in zip(offs, ns)]
    news = [N[off:off + n] for off, n in zip(offs, ns)]
    ck_old = torch.cat([bd.checksum(a).reshape(1) for a in olds])
    kw = dict(compact=compact, rice=rice)
    bound = compact or rice
    bases = ck_old if bound else None   # versions 3 and 4 are bound to checksum(old)
    # payload room from the change rate (the worst-case bound of a 30B checkpoint would not fit
    # beside it); a tensor that needs more reports its size and the batch is run again
    caps = [_cap_estimate(s) for s in specs]
    comp = bd.CompressBatch(olds, news, caps, base_checksums=bases, **kw)
    comp.run()
    torch.cuda.synchronize()
    if int(comp.status.item()) == bd.ERR_CAPACITY:
        need = [int(v) for v in comp.sizes.tolist()]
        del comp
        comp = bd.CompressBatch(olds, news, need, base_checksums=bases, **kw)
        comp.run()
        torch.cuda.synchronize()
    assert int(comp.status.item()) == bd.OK
    sizes = [int(v) for v in comp.sizes.tolist()]
    cks = bd.u64(comp.checksums)

    # sampled tensors against the oracle, byte for byte
    ck_old_list = bd.u64(ck_old)
    for i in sample:
        if bound:
            ref, ref_ck = oracle.encode(to_np_u16(olds[i]), to_np_u16(news[i]),
                                        base=ck_old_list[i], **kw)
        else:
            ref, ref_ck = oracle_pair(olds[i], news[i])
        assert sizes[i] == ref.size, specs[i].name
        assert cks[i] == ref_ck, specs[i].name
        got = comp.payloads[i][:sizes[i]].cpu().numpy()
        assert np.array_equal(got, ref), specs[i].name

    # every tensor: in-place apply restores new, applying again with checksum(old) restores old
    R = O.clone()
    rolls = [R[off:off + n] for off, n in zip(offs, ns)]
    fwd = bd.DecompressBatch(rolls, comp.payloads, sizes, comp.checksums)
    fwd.run()
    torch.cuda.synchronize()
    assert int(fwd.status.item()) == bd.OK
    assert all(int(s) == bd.OK for s in fwd.statuses.tolist())
    assert torch.equal(R.view(torch.int16), N.view(torch.int16))
    back = bd.DecompressBatch(rolls, comp.payloads, sizes, ck_old)
    back.run()
    torch.cuda.synchronize()
    assert int(back.status.item()) == bd.OK
    assert torch.equal(R.view(torch.int16), O.view(torch.int16))

    # incremental verification: forward from the checksums of old, then back from those of new
    inc = bd.IncrementalBatch(rolls, comp.payloads, sizes, ck_old, comp.checksums)
    inc.run()
    torch.cuda.synchronize()
    assert int(inc.status.item()) == bd.OK
    assert bd.u64(inc.checksums) == cks
    assert torch.equal(R.view(torch.int16), N.view(torch.int16))
    back_payloads, back_sizes = comp.payloads, sizes
    if bound:
        # a payload bound to checksum(old) is refused from new, leaving the weights alone; the
        # way back is the reverse update's payload, bound to checksum(new)
        refused = bd.IncrementalBatch(rolls, comp.payloads, sizes, comp.checksums, ck_old)
        refused.run()
        torch.cuda.synchronize()
        assert all(int(s) == bd.ERR_BASE for s in refused.statuses.tolist())
        assert torch.equal(R.view(torch.int16), N.view(torch.int16))
        comp.workspace = None   # (the forward compress is done: room for the reverse one)
        torch.cuda.empty_cache()
        rev = bd.CompressBatch(news, olds, sizes, base_checksums=comp.checksums, **kw)
        rev.run()
        torch.cuda.synchronize()
        assert int(rev.status.item()) == bd.OK
        assert [int(v) for v in rev.sizes.tolist()] == sizes
        back_payloads = rev.payloads
    inc_back = bd.IncrementalBatch(rolls, back_payloads, back_sizes, comp.checksums, ck_old)
    inc_back.run()
    torch.cuda.synchronize()
    assert int(inc_back.status.item()) == bd.OK
    assert bd.u64(inc_back.checksums) == bd.u64(ck_old)
    assert torch.equal(R.view(torch.int16), O.view(torch.int16))


def test_dense7b_full_size_batched():
    specs = W.dense7b()
    names = {s.name: i for i, s in enumerate(specs)}
    sample = [names[x] for x in ("embed", "layers.0.q", "layers.0.gate", "layers.0.down",
                                 "layers.0.norm1", "layers.31.up", "norm", "lm_head")]
    _check_workload(specs, sample)


def test_dense7b_full_size_compact():
    """The same checkpoint in version 3 (compact position blocks), bound to checksum(old)."""
    specs = W.dense7b()
    names = {s.name: i for i, s in enumerate(specs)}
    sample = [names[x] for x in ("embed", "layers.0.q", "layers.0.down", "layers.0.norm1",
                                 "norm", "lm_head")]
    _check_workload(specs, sample, compact=True)


def test_dense7b_full_size_rice():
    """The same checkpoint in version 4 (Rice-coded compact position blocks)."""
    specs = W.dense7b()
    names = {s.name: i for i, s in enumerate(specs)}
    sample = [names[x] for x in ("embed", "layers.0.k", "layers.0.up", "layers.0.norm2",
                                 "layers.31.o", "norm")]
    _check_workload(specs, sample, rice=True)


def test_moe30b_full_size_compact():
    """The MoE checkpoint in version 3: hot experts with dense chunks (version-1 bitmaps and
    compact chunks of 253..508 changes through the dense emit) beside sparse cold experts."""
    specs = W.moe30b()
    names = {s.name: i for i, s in enumerate(specs)}
    hot = max(range(len(specs)), key=lambda i: specs[i].rate)
    sample = [names["embed"], hot, names["layers.0.q"], names["lm_head"]]
    _check_workload(specs, sample, compact=True)


def test_moe30b_full_size_batched():
    specs = W.moe30b()
    names = {s.name: i for i, s in enumerate(specs)}
    hot = max(range(len(specs)), key=lambda i: specs[i].rate)   # a hot expert (bitmap chunks)
    cold = next(i for i, s in enumerate(specs) if ".experts." in s.name and s.rate < specs[hot].rate)
    sample = [names["embed"], hot, cold, names["layers.0.q"], names["layers.0.k"],
              names["layers.47.router"], names["lm_head"]]
    _check_workload(specs, sample)
