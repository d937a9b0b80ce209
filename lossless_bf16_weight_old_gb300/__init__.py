"""libbf16delta: lossless delta sync of BF16 weights on one GB300 (sm_103a).

Thin Python binding over the C ABI in include/bf16delta.h.  Every step of compress and apply
runs in the library's CUDA kernels; this module only marshals arguments and allocates device
buffers with PyTorch.

The high-level calls mirror the API listing of "Every byte counts: ARCv3 and the case for
cross-region RL":

    compressed_diff, checksum = delta_compress(src=src, dst=dst)
    restored = delta_decompress(src=src, compressed_diff=compressed_diff, checksum=checksum)
    assert torch.equal(restored.view(torch.uint8), dst.view(torch.uint8))
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import torch

from . import _lib

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_FORMAT, ERR_CHECKSUM, ERR_CUDA, ERR_BASE = range(7)
FORMAT_NAME = "bf16_xor_v1"
CHUNK_ELEMS = 4096
HEADER_BYTES = 64
_U64 = (1 << 64) - 1

__all__ = [
    "delta_compress", "delta_decompress", "compress", "decompress", "compress_batch",
    "decompress_batch", "decompress_incremental", "IncrementalBatch", "checksum",
    "compress_bound", "compress_workspace_size", "decompress_workspace_size", "payload_info",
    "DeltaError", "status_name", "MappedHostBuffer", "StreamedDecompressBatch",
]


class DeltaError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = int(code)
        super().__init__(f"{what}: {status_name(code)} ({code})" if what else status_name(code))


def status_name(code: int) -> str:
    return _lib.load().bd_status_string(int(code)).decode()


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise DeltaError(rc, what)


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _bits(t: torch.Tensor, name: str) -> tuple[int, int]:
    if t.element_size() != 2:
        raise TypeError(f"{name} must hold 16-bit values (bfloat16 bit patterns), got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr(), t.numel()


def _addr(payload) -> int:
    """Device address of a payload: a CUDA uint8 tensor, or an int address the device can read
    (for example MappedHostBuffer.device_ptr plus an offset)."""
    if isinstance(payload, torch.Tensor):
        if not payload.is_cuda:
            raise ValueError("a payload tensor must be a CUDA tensor; for host memory pass a "
                             "MappedHostBuffer device address")
        return payload.data_ptr()
    return int(payload)


_cudart_lib = None


def _cudart():
    """The CUDA runtime library, loaded once (used only for mapped host allocations)."""
    global _cudart_lib
    if _cudart_lib is None:
        for name in ("libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so.13", "libcudart.so"):
            try:
                _cudart_lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if _cudart_lib is None:
            raise RuntimeError("the CUDA runtime library was not found")
    return _cudart_lib


class MappedHostBuffer:
    """Pinned host memory mapped into the device's address space (cudaHostAlloc with
    cudaHostAllocMapped).  Kernels read it over the CPU-GPU link through `device_ptr`; host
    code fills it through `numpy()`.  A payload received into such a buffer can be applied
    without a separate host-to-device copy: pass `device_ptr + offset` as the payload."""

    _MAPPED = 0x02   # cudaHostAllocMapped

    def __init__(self, nbytes: int):
        rt = _cudart()
        self.nbytes = int(nbytes)
        self._host = ctypes.c_void_p()
        rc = rt.cudaHostAlloc(ctypes.byref(self._host), ctypes.c_size_t(max(self.nbytes, 1)),
                              ctypes.c_uint(self._MAPPED))
        if rc != 0:
            self._host = None
            raise RuntimeError(f"cudaHostAlloc failed ({rc})")
        dev = ctypes.c_void_p()
        rc = rt.cudaHostGetDevicePointer(ctypes.byref(dev), self._host, ctypes.c_uint(0))
        if rc != 0:
            rt.cudaFreeHost(self._host)
            self._host = None
            raise RuntimeError(f"cudaHostGetDevicePointer failed ({rc})")
        self.device_ptr = int(dev.value)
        self.host_ptr = int(self._host.value)

    def numpy(self):
        import numpy as np
        buf = (ctypes.c_uint8 * max(self.nbytes, 1)).from_address(self._host.value)
        return np.frombuffer(buf, dtype=np.uint8, count=self.nbytes)

    def __del__(self):
        if getattr(self, "_host", None):
            _cudart().cudaFreeHost(self._host)
            self._host = None


def _u64_tensor(values, device) -> torch.Tensor:
    vals = [int(v) & _U64 for v in values]
    vals = [v - (1 << 64) if v >= (1 << 63) else v for v in vals]
    return torch.tensor(vals, dtype=torch.int64, device=device)


def u64(t: torch.Tensor) -> list[int]:
    """Reads an int64 tensor holding unsigned 64-bit values back as Python ints."""
    return [int(v) & _U64 for v in t.reshape(-1).tolist()]


def compress_bound(n: int) -> int:
    return int(_lib.load().bd_compress_bound(int(n)))


def _sizes_arg(ns: Sequence[int]):
    arr = (ctypes.c_uint64 * max(1, len(ns)))(*[int(n) for n in ns])
    return arr, len(ns)


def compress_workspace_size(ns: Sequence[int]) -> int:
    arr, k = _sizes_arg(ns)
    return int(_lib.load().bd_compress_workspace_size(arr, k))


def decompress_workspace_size(ns: Sequence[int]) -> int:
    arr, k = _sizes_arg(ns)
    return int(_lib.load().bd_decompress_workspace_size(arr, k))


def _workspace(nbytes: int, device, workspace) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: need {nbytes} bytes")
        return workspace
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


FORMAT_OVERWRITE = 0x100   # BD_FORMAT_OVERWRITE


def _format_arg(compact: bool, overwrite: bool, rice: bool = False) -> int:
    """The format argument of bd_compress_versioned(_batch)."""
    if compact and rice:
        raise ValueError("compact (version 3) and rice (version 4) exclude each other")
    return (4 if rice else 3 if compact else 2) | (FORMAT_OVERWRITE if overwrite else 0)


def compress(old: torch.Tensor, new: torch.Tensor, *, payload: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None, base_checksum=None, compact: bool = False,
             overwrite: bool = False, rice: bool = False, stream=None):
    """Encodes old -> new on the GPU.  Returns device tensors
    (payload uint8[cap], size int64[1], checksum int64[1] (unsigned bits), status int32[1]),
    all written asynchronously on the stream.  With base_checksum (an int or int64[1] device
    tensor: the checksum of old as the caller knows it) the payload is bound to that base
    (bd_compress_versioned): version 2, version 3 (compact position blocks) when `compact` is
    set, or version 4 (Rice-coded compact position blocks) when `rice` is set; with
    `overwrite` the payload carries new values instead of XOR masks (applying it again, to
    weights it has wholly or partly updated, gives the same result)."""
    if (compact or overwrite or rice) and base_checksum is None:
        raise ValueError("compact, Rice and overwrite payloads are bound to a base: "
                         "pass base_checksum")
    fmt = _format_arg(compact, overwrite, rice)
    po, n = _bits(old, "old")
    pn, n2 = _bits(new, "new")
    if n != n2:
        raise ValueError("old and new must have the same number of elements")
    dev = old.device
    if payload is None:
        payload = torch.empty(compress_bound(n), dtype=torch.uint8, device=dev)
    ws = _workspace(compress_workspace_size([n]), dev, workspace)
    size = torch.empty(1, dtype=torch.int64, device=dev)
    ck = torch.empty(1, dtype=torch.int64, device=dev)
    st = torch.empty(1, dtype=torch.int32, device=dev)
    if base_checksum is None:
        rc = _lib.load().bd_compress(po, pn, n, payload.data_ptr(), payload.numel(),
                                     ws.data_ptr(), ws.numel(), size.data_ptr(), ck.data_ptr(),
                                     st.data_ptr(), _stream(stream))
        _check(rc, "bd_compress")
    else:
        if not isinstance(base_checksum, torch.Tensor):
            base_checksum = _u64_tensor([base_checksum], dev)
        rc = _lib.load().bd_compress_versioned(po, pn, n, payload.data_ptr(), payload.numel(),
                                               ws.data_ptr(), ws.numel(), size.data_ptr(),
                                               ck.data_ptr(), base_checksum.data_ptr(),
                                               fmt, st.data_ptr(),
                                               _stream(stream))
        _check(rc, "bd_compress_versioned")
    return payload, size, ck, st


def decompress(old: torch.Tensor, payload: torch.Tensor, size: int, expected,
               *, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Applies payload[:size] to old (in place when out is old), verifying the checksum.
    `expected` is an int or an int64[1] device tensor.  Returns the int32[1] device status."""
    po, n = _bits(old, "old")
    if out is None:
        out = torch.empty_like(old)
    pout, n2 = _bits(out, "out")
    if n2 != n:
        raise ValueError("out must have as many elements as old")
    if not isinstance(expected, torch.Tensor):
        expected = _u64_tensor([expected], old.device)
    ws = _workspace(decompress_workspace_size([n]), old.device, workspace)
    st = torch.empty(1, dtype=torch.int32, device=old.device)
    rc = _lib.load().bd_decompress(po, n, _addr(payload), int(size), expected.data_ptr(),
                                   pout, ws.data_ptr(), ws.numel(), st.data_ptr(),
                                   _stream(stream))
    _check(rc, "bd_decompress")
    return st


def decompress_incremental(w: torch.Tensor, payload: torch.Tensor, size: int, ck_old, expected,
                           *, workspace: torch.Tensor | None = None, stream=None
                           ) -> tuple[torch.Tensor, torch.Tensor]:
    """Applies payload[:size] to w in place, verifying incrementally from ck_old, the checksum
    of w before the call (see bd_decompress_incremental).  ck_old and expected are ints or
    int64[1] device tensors.  Returns (int32[1] status, int64[1] computed checksum)."""
    pw, n = _bits(w, "w")
    if not isinstance(ck_old, torch.Tensor):
        ck_old = _u64_tensor([ck_old], w.device)
    if not isinstance(expected, torch.Tensor):
        expected = _u64_tensor([expected], w.device)
    ws = _workspace(decompress_workspace_size([n]), w.device, workspace)
    st = torch.empty(1, dtype=torch.int32, device=w.device)
    ck = torch.zeros(1, dtype=torch.int64, device=w.device)
    rc = _lib.load().bd_decompress_incremental(pw, n, _addr(payload), int(size),
                                               ck_old.data_ptr(), expected.data_ptr(),
                                               ck.data_ptr(), ws.data_ptr(), ws.numel(),
                                               st.data_ptr(), _stream(stream))
    _check(rc, "bd_decompress_incremental")
    return st, ck


def checksum(w: torch.Tensor, *, stream=None) -> torch.Tensor:
    """Checksum of a BF16 tensor as an int64[1] device tensor (unsigned bits)."""
    pw, n = _bits(w, "w")
    out = torch.empty(1, dtype=torch.int64, device=w.device)
    _check(_lib.load().bd_checksum(pw, n, out.data_ptr(), _stream(stream)), "bd_checksum")
    return out


class CompressBatch:
    """Device buffers and the C item table of one batched compress over fixed tensors."""

    def __init__(self, olds: Sequence[torch.Tensor], news: Sequence[torch.Tensor],
                 caps: Sequence[int] | None = None, base_checksums: torch.Tensor | None = None,
                 compact: bool = False, overwrite: bool = False, rice: bool = False,
                 workspace: torch.Tensor | None = None):
        """base_checksums (int64[k] device tensor, optional): payloads bound to these base
        checksums (bd_compress_versioned_batch), version 2, version 3 (compact position
        blocks) when `compact` is set or version 4 (Rice-coded ones) when `rice` is set,
        overwrite payloads when `overwrite` is set.  workspace (optional, uint8 device tensor
        of at least compress_workspace_size bytes) may be shared by batches whose runs never
        overlap on the GPU; one is allocated otherwise."""
        if (compact or overwrite or rice) and base_checksums is None:
            raise ValueError("compact, Rice and overwrite payloads are bound to a base: "
                             "pass base_checksums")
        self.format = _format_arg(compact, overwrite, rice)
        if len(olds) != len(news):
            raise ValueError("olds and news differ in length")
        k = len(olds)
        dev = olds[0].device
        ns = []
        for o, nw in zip(olds, news):
            if o.numel() != nw.numel():
                raise ValueError("old/new element counts differ")
            ns.append(o.numel())
        caps = list(caps) if caps is not None else [compress_bound(n) for n in ns]
        self.ns, self.caps = ns, caps
        offs, tot = [], 0
        for c in caps:
            offs.append(tot)
            tot += (int(c) + 255) // 256 * 256
        self.payload_buf = torch.empty(max(tot, 256), dtype=torch.uint8, device=dev)
        self.payloads = [self.payload_buf[o:o + c] for o, c in zip(offs, caps)]
        self.sizes = torch.zeros(k, dtype=torch.int64, device=dev)
        self.checksums = torch.zeros(k, dtype=torch.int64, device=dev)
        self.statuses = torch.zeros(k, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = _workspace(compress_workspace_size(ns), dev, workspace)
        items = (_lib.CompressItem * max(1, k))()
        for i in range(k):
            items[i].d_old = _bits(olds[i], "old")[0]
            items[i].d_new = _bits(news[i], "new")[0]
            items[i].n = ns[i]
            items[i].d_payload = self.payloads[i].data_ptr()
            items[i].cap = int(caps[i])
            items[i].d_size = self.sizes.data_ptr() + 8 * i
            items[i].d_checksum = self.checksums.data_ptr() + 8 * i
            items[i].d_status = self.statuses.data_ptr() + 4 * i
        self._keep = (list(olds), list(news), base_checksums)
        self.items, self.k = items, k
        self.bases = None
        if base_checksums is not None:
            self.bases = (ctypes.c_void_p * max(1, k))(
                *[base_checksums.data_ptr() + 8 * i for i in range(k)])

    def run(self, stream=None) -> None:
        if self.bases is not None:
            rc = _lib.load().bd_compress_versioned_batch(
                self.items, self.bases, self.k, self.format, self.workspace.data_ptr(),
                self.workspace.numel(), self.status.data_ptr(), _stream(stream))
            _check(rc, "bd_compress_versioned_batch")
            return
        rc = _lib.load().bd_compress_batch(self.items, self.k, self.workspace.data_ptr(),
                                           self.workspace.numel(), self.status.data_ptr(),
                                           _stream(stream))
        _check(rc, "bd_compress_batch")



def debug_compress_stall(batch: CompressBatch, stall: int, stream=None) -> None:
    """bd_debug_compress_stall on a CompressBatch of version-1 payloads: tensor `stall` is
    never published, so the persistent compress's bounded wait runs out; afterwards
    ``batch.status`` and every entry of ``batch.statuses`` hold ERR_CUDA.  Fault injection
    for tests of that error path."""
    if batch.bases is not None:
        raise ValueError("debug_compress_stall takes a batch of version-1 payloads")
    rc = _lib.load().bd_debug_compress_stall(batch.items, batch.k, int(stall),
                                             batch.workspace.data_ptr(), batch.workspace.numel(),
                                             batch.status.data_ptr(), _stream(stream))
    _check(rc, "bd_debug_compress_stall")

class DecompressBatch:
    """Device buffers and the C item table of one batched decompress over fixed tensors."""

    def __init__(self, olds: Sequence[torch.Tensor], payloads: Sequence[torch.Tensor],
                 sizes: Sequence[int], expected: torch.Tensor,
                 outs: Sequence[torch.Tensor] | None = None,
                 workspace: torch.Tensor | None = None):
        """workspace: as for CompressBatch (decompress_workspace_size bytes)."""
        k = len(olds)
        dev = olds[0].device
        outs = list(outs) if outs is not None else list(olds)
        ns = [o.numel() for o in olds]
        self.statuses = torch.zeros(k, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = _workspace(decompress_workspace_size(ns), dev, workspace)
        self.expected = expected
        items = (_lib.DecompressItem * max(1, k))()
        for i in range(k):
            items[i].d_old = _bits(olds[i], "old")[0]
            items[i].d_out = _bits(outs[i], "out")[0]
            items[i].n = ns[i]
            items[i].d_payload = _addr(payloads[i])
            items[i].size = int(sizes[i])
            items[i].d_expected = expected.data_ptr() + 8 * i
            items[i].d_status = self.statuses.data_ptr() + 4 * i
        self._keep = (list(olds), list(payloads), outs)
        self.items, self.k = items, k

    def set_expected(self, expected: torch.Tensor) -> None:
        for i in range(self.k):
            self.items[i].d_expected = expected.data_ptr() + 8 * i
        self.expected = expected

    def run(self, stream=None) -> None:
        rc = _lib.load().bd_decompress_batch(self.items, self.k, self.workspace.data_ptr(),
                                             self.workspace.numel(), self.status.data_ptr(),
                                             _stream(stream))
        _check(rc, "bd_decompress_batch")


class StreamedDecompressBatch:
    """Item table of one bd_decompress_batch_streamed call: the payloads lie in page-locked
    host memory (a MappedHostBuffer, or a pinned CPU uint8 tensor) at byte offsets `offsets`,
    and are copied through two device slots of `slot_bytes` each while the previous slot's
    tensors are applied."""

    def __init__(self, olds: Sequence[torch.Tensor], host_payloads, offsets: Sequence[int],
                 sizes: Sequence[int], expected: torch.Tensor, slot_bytes: int | None = None,
                 outs: Sequence[torch.Tensor] | None = None,
                 workspace: torch.Tensor | None = None):
        k = len(olds)
        dev = olds[0].device
        outs = list(outs) if outs is not None else list(olds)
        ns = [o.numel() for o in olds]
        if isinstance(host_payloads, MappedHostBuffer):
            host = host_payloads.host_ptr
        elif isinstance(host_payloads, torch.Tensor) and not host_payloads.is_cuda:
            host = host_payloads.data_ptr()
        else:
            raise ValueError("host_payloads must be a MappedHostBuffer or a CPU tensor")
        largest = max([(int(z) + 255) // 256 * 256 for z in sizes] + [256])
        self.slot_bytes = int(slot_bytes) if slot_bytes is not None else max(64 << 20, largest)
        self.staging = torch.empty(2 * self.slot_bytes, dtype=torch.uint8, device=dev)
        self.statuses = torch.zeros(k, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = _workspace(decompress_workspace_size(ns), dev, workspace)
        self.copy_stream = torch.cuda.Stream(device=dev)
        items = (_lib.DecompressItem * max(1, k))()
        for i in range(k):
            items[i].d_old = _bits(olds[i], "old")[0]
            items[i].d_out = _bits(outs[i], "out")[0]
            items[i].n = ns[i]
            items[i].d_payload = host + int(offsets[i])
            items[i].size = int(sizes[i])
            items[i].d_expected = expected.data_ptr() + 8 * i
            items[i].d_status = self.statuses.data_ptr() + 4 * i
        self._keep = (list(olds), host_payloads, outs, expected)
        self.items, self.k = items, k

    def run(self, stream=None, copy_stream=None) -> None:
        cs = copy_stream if copy_stream is not None else self.copy_stream
        rc = _lib.load().bd_decompress_batch_streamed(
            self.items, self.k, self.staging.data_ptr(), self.slot_bytes,
            self.workspace.data_ptr(), self.workspace.numel(), self.status.data_ptr(),
            _stream(stream), _stream(cs))
        _check(rc, "bd_decompress_batch_streamed")


class IncrementalBatch:
    """Item table of one batched incremental apply over fixed tensors (in place)."""

    def __init__(self, ws: Sequence[torch.Tensor], payloads: Sequence[torch.Tensor],
                 sizes: Sequence[int], ck_old: torch.Tensor, expected: torch.Tensor,
                 workspace: torch.Tensor | None = None):
        """workspace: as for CompressBatch (decompress_workspace_size bytes)."""
        k = len(ws)
        dev = ws[0].device
        ns = [w.numel() for w in ws]
        self.statuses = torch.zeros(k, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.checksums = torch.zeros(k, dtype=torch.int64, device=dev)
        self.workspace = _workspace(decompress_workspace_size(ns), dev, workspace)
        items = (_lib.IncrementalItem * max(1, k))()
        for i in range(k):
            items[i].d_w = _bits(ws[i], "w")[0]
            items[i].n = ns[i]
            items[i].d_payload = _addr(payloads[i])
            items[i].size = int(sizes[i])
            items[i].d_ck_old = ck_old.data_ptr() + 8 * i
            items[i].d_expected = expected.data_ptr() + 8 * i
            items[i].d_ck_out = self.checksums.data_ptr() + 8 * i
            items[i].d_status = self.statuses.data_ptr() + 4 * i
        self._keep = (list(ws), list(payloads), ck_old, expected)
        self.items, self.k = items, k

    def run(self, stream=None) -> None:
        rc = _lib.load().bd_decompress_incremental_batch(
            self.items, self.k, self.workspace.data_ptr(), self.workspace.numel(),
            self.status.data_ptr(), _stream(stream))
        _check(rc, "bd_decompress_incremental_batch")


def compress_batch(olds, news, caps=None, stream=None) -> CompressBatch:
    b = CompressBatch(olds, news, caps)
    b.run(stream)
    return b


def decompress_batch(olds, payloads, sizes, expected, outs=None, stream=None) -> DecompressBatch:
    b = DecompressBatch(olds, payloads, sizes, expected, outs)
    b.run(stream)
    return b


def payload_info(header: bytes) -> dict:
    """Parses a payload header held in host memory."""
    info = _lib.PayloadInfo()
    buf = (ctypes.c_uint8 * len(header)).from_buffer_copy(header)
    _check(_lib.load().bd_payload_info(buf, len(header), ctypes.byref(info)), "bd_payload_info")
    return {f: getattr(info, f) for f, _ in _lib.PayloadInfo._fields_}


def _format(compression_format: str) -> None:
    if compression_format != FORMAT_NAME:
        raise ValueError(f"unsupported compression_format {compression_format!r}; "
                         f"this library implements {FORMAT_NAME!r}")


def delta_compress(src: torch.Tensor, dst: torch.Tensor,
                   compression_format: str = FORMAT_NAME) -> tuple[torch.Tensor, int]:
    """Returns (compressed_diff: uint8 device tensor, checksum of dst as an int)."""
    _format(compression_format)
    payload, size, ck, st = compress(src.reshape(-1), dst.reshape(-1))
    sz, c, s = int(size.item()), u64(ck)[0], int(st.item())
    _check(s, "delta_compress")
    return payload[:sz], c


def delta_decompress(src: torch.Tensor, compressed_diff: torch.Tensor, checksum: int,
                     compression_format: str = FORMAT_NAME) -> torch.Tensor:
    """Returns a new tensor holding src with the delta applied; raises DeltaError when the
    payload is malformed or the checksum does not match."""
    _format(compression_format)
    out = torch.empty_like(src)
    st = decompress(src.reshape(-1), compressed_diff, compressed_diff.numel(), checksum,
                    out=out.reshape(-1))
    _check(int(st.item()), "delta_decompress")
    return out
