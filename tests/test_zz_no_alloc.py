"""bd_decompress_noalloc against bd_decompress (GPU).

bd_decompress_noalloc serves callers that cannot allocate device memory, such as an
inference engine whose allocator already holds nearly all of HBM for weights and KV cache.
It takes no workspace: its scratch is a fixed array inside the library.  Here it must give
exactly what the workspace entry point gives (integer work, tolerance 0): the same restored
weights and the same status, on two calls in a row (the second call finds the first call's
contents in the shared scratch array).

This file is named to be collected last, so that a run stopping at the first failure has
already run every other test.  It passes alone in a fresh process as well.
"""
import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

bd = pytest.importorskip("lossless_bf16_weight_old_gb300")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return bd._lib.load()


def _noalloc(lib, old, payload, size, expected, out):
    st = torch.full((1,), -1, dtype=torch.int32, device=old.device)
    rc = lib.bd_decompress_noalloc(old.data_ptr(), old.numel(), payload.data_ptr(), int(size),
                                   expected.data_ptr(), out.data_ptr(), st.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == bd.OK
    return st


@pytest.mark.parametrize("call", [0, 1])
def test_noalloc_matches_workspace_entry_point(lib, call):
    # two calls in a row, on different tensors (sizes, densities, a ragged last chunk)
    spec = [W.Spec("a", (3 * 4096 * 64 + 1234,), rate=0.02, tid=41),
            W.Spec("b", (4096 * 300 + 7,), rate=0.3, tid=42)][call]
    old, new = W.make_pair(spec, device="cuda")
    payload, size_t, ck, st = bd.compress(old, new)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    size = int(size_t.item())

    ref = torch.empty_like(old)
    st_ref = bd.decompress(old, payload, size, ck, out=ref)
    got = torch.empty_like(old)
    st_got = _noalloc(lib, old, payload, size, ck, got)
    torch.cuda.synchronize()
    assert int(st_ref.item()) == int(st_got.item()) == bd.OK
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(got.view(torch.int16), new.view(torch.int16))

    # in place, and a wrong expected checksum: same status as the workspace entry point
    work = old.clone()
    st_in = _noalloc(lib, work, payload, size, ck, work)
    bad_ck = ck ^ 1
    st_bad = _noalloc(lib, old, payload, size, bad_ck, torch.empty_like(old))
    st_bad_ref = bd.decompress(old, payload, size, bad_ck, out=torch.empty_like(old))
    torch.cuda.synchronize()
    assert int(st_in.item()) == bd.OK
    assert torch.equal(work.view(torch.int16), new.view(torch.int16))
    assert int(st_bad.item()) == int(st_bad_ref.item()) == bd.ERR_CHECKSUM


def test_noalloc_empty_tensor(lib):
    # n = 0: the 64-byte header alone, checksum 0; twice in a row, as above
    old = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    payload, size_t, ck, st = bd.compress(old, old)
    torch.cuda.synchronize()
    assert int(st.item()) == bd.OK
    size = int(size_t.item())
    for _ in range(2):
        out = torch.empty_like(old)
        st_ref = bd.decompress(old, payload, size, ck, out=out)
        st_got = _noalloc(lib, old, payload, size, ck, out)
        st_bad = _noalloc(lib, old, payload, size, ck ^ 1, out)
        torch.cuda.synchronize()
        assert int(st_ref.item()) == int(st_got.item()) == bd.OK
        assert int(st_bad.item()) == bd.ERR_CHECKSUM


def test_noalloc_rejects_tensors_beyond_its_scratch(lib):
    limit = 1 << 27
    dummy = ctypes.c_void_p(1 << 20)
    rc = lib.bd_decompress_noalloc(dummy, limit + 1, dummy, 64, dummy, dummy, dummy, None)
    assert rc == bd.ERR_INVALID_ARG
