"""Host <-> device helpers for the GPU parity tests (bit-exact transfers)."""
import numpy as np
import torch

_SIGNED = {np.dtype(np.uint32): np.int32, np.dtype(np.uint64): np.int64,
           np.dtype(np.uint16): np.int16}


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(_SIGNED.get(a.dtype, a.dtype))).cuda()


def to_host(t: torch.Tensor, dtype) -> np.ndarray:
    return t.cpu().numpy().view(dtype)


def poisoned_like(t: torch.Tensor) -> torch.Tensor:
    """An output buffer filled with 0xAA bytes, so unwritten slots show up."""
    out = torch.empty_like(t)
    out.view(torch.uint8).fill_(0xAA)
    return out


def field(keys: np.ndarray, begin: int, end: int) -> np.ndarray:
    keys = keys.astype(np.uint64)
    w = end - begin
    mask = np.uint64((1 << w) - 1) if w < 64 else np.uint64(0xFFFFFFFFFFFFFFFF)
    return (keys >> np.uint64(begin)) & mask
