"""Helpers shared by the GPU tests: conversions between torch tensors and the oracle's
numpy arrays (no arithmetic of the method here)."""
import numpy as np
import torch

import oracle


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16)


def from_np_u16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def oracle_pair(old: torch.Tensor, new: torch.Tensor):
    """Oracle payload bytes and checksum for device tensors old/new."""
    return oracle.encode(to_np_u16(old), to_np_u16(new))


def u64(v: int) -> int:
    return int(v) & ((1 << 64) - 1)
