"""Parity at full size on the 7B-shaped dense checkpoint and the 30B-shaped MoE checkpoint, in
the launch configuration the benchmark times: one batched compress over every tensor of the
checkpoint (held in one flat buffer per checkpoint, tensors at 256-byte aligned offsets), then
one batched in-place apply on a copy of old; both checkpoints in version 1, version 3 (compact
position blocks) and version 4 (Rice-coded compact position blocks).

The oracle checks EVERY tensor of the checkpoint one by one: payload bytes, size and checksum
(integer work, tolerance 0).  Byte equality matters beyond "restored == new" because the
decoders of versions 3 and 4 accept codings the encoder never writes (another Rice parameter,
a chunk kept on version-1 blocks), so a wrong choice would still restore.  The oracle runs
one tensor per host thread (its C calls release the interpreter lock), fed by device-to-host
copies of one tensor at a time with a bound on the host memory in flight.  Every tensor is
also checked by properties of the apply: each status is OK, the restored checkpoint equals new
bit for bit, and applying the same payloads again with the checksums of old restores old.
"""
import collections
import os
from concurrent.futures import ThreadPoolExecutor

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


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_one(name, o, nw, got, ck, base, kw):
    """The oracle's payload for one tensor, compared with the GPU's (a message, or None)."""
    ref, ref_ck = oracle.encode(o, nw, base=base, cap=got.size, **kw)
    if ref.size != got.size:
        return f"{name}: size {got.size} != oracle {ref.size}"
    if ref_ck != ck:
        return f"{name}: checksum {ck:#x} != oracle {ref_ck:#x}"
    if not np.array_equal(ref, got):
        at = int(np.flatnonzero(ref != got)[0])
        return f"{name}: payload differs from the oracle's first at byte {at}"
    return None


def _oracle_every_tensor(specs, olds, news, payloads, sizes, cks, bases, kw):
    """Compares every tensor's payload, size and checksum with the oracle's, one tensor per
    host thread; at most `limit` bytes of host copies are in flight."""
    largest = max(4 * s.numel for s in specs)
    limit = max(6 << 30, 3 * largest)
    pending = collections.deque()
    in_flight = 0
    errors = []
    checked = 0

    def drain_one():
        nonlocal in_flight, checked
        fut, nbytes = pending.popleft()
        msg = fut.result()
        in_flight -= nbytes
        checked += 1
        if msg is not None:
            errors.append(msg)

    with ThreadPoolExecutor(max_workers=min(_host_cores(), 64)) as ex:
        for i, s in enumerate(specs):
            nbytes = 4 * s.numel + sizes[i]
            while pending and in_flight + nbytes > limit:
                drain_one()
            o, nw = to_np_u16(olds[i]), to_np_u16(news[i])
            got = payloads[i][:sizes[i]].cpu().numpy()
            base = None if bases is None else bases[i]
            pending.append((ex.submit(_oracle_one, s.name, o, nw, got, cks[i], base, kw), nbytes))
            in_flight += nbytes
        while pending:
            drain_one()
    assert checked == len(specs)
    assert not errors, f"{len(errors)} of {len(specs)} tensors differ: {errors[:5]}"


def _check_workload(specs, compact=False, rice=False):
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

    # every tensor against the oracle, byte for byte
    _oracle_every_tensor(specs, olds, news, comp.payloads, sizes, cks,
                         bd.u64(ck_old) if bound else None, kw)

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
    _check_workload(W.dense7b())


def test_dense7b_full_size_compact():
    """The same checkpoint in version 3 (compact position blocks), bound to checksum(old)."""
    _check_workload(W.dense7b(), compact=True)


def test_dense7b_full_size_rice():
    """The same checkpoint in version 4 (Rice-coded compact position blocks)."""
    _check_workload(W.dense7b(), rice=True)


def test_moe30b_full_size_batched():
    """The MoE checkpoint: hot experts with dense chunks (bitmaps, the dense emit and apply)
    beside sparse cold experts, attention, routers, embedding and head."""
    _check_workload(W.moe30b())


def test_moe30b_full_size_compact():
    """The MoE checkpoint in version 3: compact chunks of 253..508 changes through the dense
    emit beside version-1 bitmaps."""
    _check_workload(W.moe30b(), compact=True)


def test_moe30b_full_size_rice():
    """The MoE checkpoint in version 4."""
    _check_workload(W.moe30b(), rice=True)
