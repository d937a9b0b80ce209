"""A single tensor past 2^32 elements (GPU): the 64-bit index paths at the largest sizes this
test can hold (about 30 GB on the device).

At this size the oracle is not run on the whole tensor; the payload is checked through
properties that fix it at any size, each computed independently of the library's kernels:
  - the header's n, C, sum M, sum R equal the class counts of old ^ new computed with torch;
  - the whole per-chunk count table equals the per-chunk class counts computed with torch;
  - the payload size equals the closed form 64 + 4C + 2 sum R + sum_c (blk(M_c) + blk(R_c))
    + ceil(7 sum M / 8), with blk(k) = 2k if 2k < ceil(L/8) else ceil(L/8);
  - the checksum returned by compress equals the standalone checksum kernel's on new;
  - the apply restores new bit for bit and verifies; the incremental apply back restores old.
"""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")

N = (1 << 32) + 12345
CHUNK = 4096


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    torch.cuda.empty_cache()   # blocks cached by earlier tests count as used otherwise
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * (1 << 30):
        pytest.skip("needs about 40 GB of free device memory")
    bd._lib.load()


def _counts(old, new):
    """Per-chunk (M, R) counts of old ^ new, with torch (no library code), in pieces of 2^28
    elements (whole chunks) to bound the temporaries."""
    C = (N + CHUNK - 1) // CHUNK
    m = torch.empty(C, dtype=torch.int64, device="cuda")
    r = torch.empty_like(m)
    step = 1 << 28
    for a in range(0, N, step):
        b = min(N, a + step)
        x = (old[a:b].view(torch.int16) ^ new[a:b].view(torch.int16)).to(torch.int32) & 0xFFFF
        c0, nc = a // CHUNK, (b - a + CHUNK - 1) // CHUNK
        pad = nc * CHUNK - (b - a)
        ch = torch.nn.functional.pad((x != 0).to(torch.int32), (0, pad)).view(nc, CHUNK).sum(1)
        rr = torch.nn.functional.pad(((x & 0xFF80) != 0).to(torch.int32),
                                     (0, pad)).view(nc, CHUNK).sum(1)
        m[c0:c0 + nc] = ch - rr
        r[c0:c0 + nc] = rr
        del x
    return m, r


def test_tensor_past_2_pow_32_elements():
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    old = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    for a in range(0, N, 1 << 28):   # fill in pieces to bound the temporaries
        b = min(N, a + (1 << 28))
        old[a:b] = (torch.randn(b - a, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    new = old.clone()
    for a in range(0, N, 1 << 28):
        b = min(N, a + (1 << 28))
        new[a:b] = W.mutate(old[a:b], 0.002, g)
    m, r = _counts(old, new)
    C = m.numel()

    cap = 64 + 4 * C + 2 * int(r.sum()) + 2 * (2 * int((m + r).sum())) + 2 * CHUNK // 8 * 4 + 64
    payload = torch.empty(cap, dtype=torch.uint8, device="cuda")
    payload, size, ck, st = bd.compress(old, new, payload=payload)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    size = int(size.item())

    info = bd.payload_info(payload[:64].cpu().numpy().tobytes())
    assert info["n"] == N and info["chunks"] == C
    assert info["n_mant"] == int(m.sum()) and info["n_rare"] == int(r.sum())
    table = payload[64:64 + 4 * C].view(torch.int16).view(C, 2).to(torch.int64) & 0xFFFF
    assert torch.equal(table[:, 0], m) and torch.equal(table[:, 1], r)

    L = torch.full((C,), CHUNK, dtype=torch.int64, device="cuda")
    L[-1] = N - (C - 1) * CHUNK
    B = (L + 7) // 8
    blk = lambda k: torch.where(2 * k < B, 2 * k, B)
    closed = 64 + 4 * C + 2 * int(r.sum()) + int((blk(m) + blk(r)).sum()) + (7 * int(m.sum()) + 7) // 8
    assert size == closed == info["total_size"]

    assert bd.u64(ck) == bd.u64(bd.checksum(new))

    out = torch.empty_like(old)
    st2 = bd.decompress(old, payload, size, ck, out=out)
    torch.cuda.synchronize()
    assert int(st2.item()) == bd.OK
    assert torch.equal(out.view(torch.int16), new.view(torch.int16))
    del out

    w = new.clone()
    del new
    st3, ck3 = bd.decompress_incremental(w, payload, size, ck, bd.checksum(old))
    torch.cuda.synchronize()
    assert int(st3.item()) == bd.OK
    assert bd.u64(ck3) == bd.u64(bd.checksum(old))
    assert torch.equal(w.view(torch.int16), old.view(torch.int16))
