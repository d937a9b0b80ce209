"""The bounded wait of the persistent compress (GPU).

In the batched compress of version-1 payloads a warp that is to emit a tensor waits until the
tensor's last batch is counted.  The schedule guarantees that the wait ends; the wait is also
bounded (about a second of idle polling), after which the kernel reports BD_ERR_CUDA and
returns.  The fault-injection hook keeps one tensor of the call from ever being published (a
flag that nothing sets), so the bound runs out: the call must end on its own, report
BD_ERR_CUDA for the call and for every tensor, and leave the CUDA context and the workspace
fit for the next call, whose payloads must be the oracle's.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import from_np_u16, u64

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    bd._lib.load()


def _pairs(seed, sizes, rate=0.02):
    rng = np.random.default_rng(seed)
    out = []
    for n in sizes:
        o = rng.integers(0, 1 << 16, n, dtype=np.uint16)
        nw = o.copy()
        pick = rng.random(n) < rate
        nw[pick] ^= rng.integers(1, 1 << 16, int(pick.sum())).astype(np.uint16)
        out.append((o, nw))
    return out


@pytest.mark.parametrize("stall", [0, 1, 2])
def test_stalled_tensor_gives_up_and_reports(stall):
    pairs = _pairs(40 + stall, [4096 * 5 + 7, 4096 * 3, 100])
    olds = [from_np_u16(p[0]) for p in pairs]
    news = [from_np_u16(p[1]) for p in pairs]
    cb = bd.CompressBatch(olds, news)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    bd.debug_compress_stall(cb, stall)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(cb.status.item()) == bd.ERR_CUDA
    assert [int(v) for v in cb.statuses.tolist()] == [bd.ERR_CUDA] * 3
    assert 0.05 < elapsed < 30, elapsed   # the bound ran out, and ended the call
    # the context and the same workspace serve the next call
    cb.run()
    torch.cuda.synchronize()
    assert int(cb.status.item()) == bd.OK
    for i, (o, nw) in enumerate(pairs):
        ref, ck = oracle.encode(o, nw)
        n = int(cb.sizes[i].item())
        assert np.array_equal(cb.payloads[i][:n].cpu().numpy(), ref), i
        assert u64(cb.checksums[i].item()) == ck, i


def test_hook_refuses_a_call_without_the_persistent_compress():
    # one tensor of 2^24 + 4096 elements: 4097 one-chunk batches, more than the persistent
    # compress takes, so the call would take the separate kernels, which do not wait
    n = (1 << 24) + 4096
    o = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    cb = bd.CompressBatch([o], [o.clone()])
    with pytest.raises(bd.DeltaError):
        bd.debug_compress_stall(cb, 0)
    cb.run()
    torch.cuda.synchronize()
    assert int(cb.status.item()) == bd.OK
