"""Apply from a payload held in host memory (GPU).

The payload is placed in pinned host memory mapped into the device's address space
(MappedHostBuffer: cudaHostAlloc with cudaHostAllocMapped, device address from
cudaHostGetDevicePointer); the apply kernels read it over the CPU-GPU link with no separate
host-to-device copy.  Results must be identical to the oracle's (integer work, tolerance 0)
for the full and the incremental apply, single and batched.
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


def test_single_apply_from_host_payload():
    old, new = W.make_pair(W.Spec("h", (4096 * 150 + 777,), rate=0.02, tid=12), device="cuda")
    old, new = old.reshape(-1), new.reshape(-1)
    ref, ck = oracle_pair(old, new)
    buf = bd.MappedHostBuffer(ref.size)
    buf.numpy()[:] = ref
    out = torch.empty_like(old)
    st = bd.decompress(old, buf.device_ptr, ref.size, ck, out=out)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    st_ref, restored = oracle.decode(to_np_u16(old), ref, ck)
    assert st_ref == oracle.OK
    assert np.array_equal(to_np_u16(out), restored)
    # in place, incremental, from the same host payload
    w = old.clone()
    st2, ck2 = bd.decompress_incremental(w, buf.device_ptr, ref.size,
                                         oracle.checksum(to_np_u16(old)), ck)
    torch.cuda.synchronize()
    assert int(st2.item()) == bd.OK and bd.u64(ck2)[0] == ck
    assert torch.equal(w.view(torch.int16), new.view(torch.int16))


def test_batched_apply_from_host_payloads():
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    sizes = [4096 * 64, 12345, 1, 4096 * 3 + 5, 70001]
    rates = [0.02, 0.3, 0.0, 1.0, 0.05]
    olds, news, refs, cks = [], [], [], []
    for n, r in zip(sizes, rates):
        o = (torch.randn(n, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        nw = W.mutate(o, r, g)
        ref, ck = oracle_pair(o, nw)
        olds.append(o)
        news.append(nw)
        refs.append(ref)
        cks.append(ck)
    offs, tot = [], 0
    for r in refs:
        offs.append(tot)
        tot += (r.size + 255) // 256 * 256
    buf = bd.MappedHostBuffer(tot)
    host = buf.numpy()
    for r, o in zip(refs, offs):
        host[o:o + r.size] = r
    outs = [torch.empty_like(o) for o in olds]
    b = bd.DecompressBatch(olds, [buf.device_ptr + o for o in offs], [r.size for r in refs],
                           bd._u64_tensor(cks, "cuda"), outs=outs)
    b.run()
    torch.cuda.synchronize()
    assert int(b.status.item()) == bd.OK
    for o, nw in zip(outs, news):
        assert torch.equal(o.view(torch.int16), nw.view(torch.int16))


@pytest.mark.parametrize("version", [3, 4])
@pytest.mark.parametrize("overwrite", [False, True])
def test_versioned_payloads_from_host_memory(overwrite, version):
    """Version-3 and version-4 payloads (XOR and overwrite) read from mapped host memory by the
    full, the incremental and the no-workspace apply: the oracle's result in every case."""
    old, new = W.make_pair(W.Spec("h3", (4096 * 90 + 321,), rate=0.04, tid=13), device="cuda")
    old, new = old.reshape(-1), new.reshape(-1)
    o, nw = to_np_u16(old), to_np_u16(new)
    base = oracle.checksum(o)
    ref, ck = oracle.encode(o, nw, base=base, compact=version == 3, rice=version == 4,
                            overwrite=overwrite)
    buf = bd.MappedHostBuffer(ref.size)
    buf.numpy()[:] = ref
    out = torch.empty_like(old)
    st = bd.decompress(old, buf.device_ptr, ref.size, ck, out=out)
    w = old.clone()
    st2, ck2 = bd.decompress_incremental(w, buf.device_ptr, ref.size, base, ck)
    lib = bd._lib.load()
    out3 = torch.empty_like(old)
    st3 = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ckt = bd._u64_tensor([ck], "cuda")
    assert lib.bd_decompress_noalloc(old.data_ptr(), old.numel(), buf.device_ptr, ref.size,
                                     ckt.data_ptr(), out3.data_ptr(), st3.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream) == bd.OK
    torch.cuda.synchronize()
    assert int(st.item()) == int(st2.item()) == int(st3.item()) == bd.OK
    assert bd.u64(ck2)[0] == ck
    for r in (out, w, out3):
        assert torch.equal(r.view(torch.int16), new.view(torch.int16))
