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


def assert_pairs(got_keys, got_vals, want_keys, want_vals, what: str = ""):
    """Element-by-element parity of a key-value sort with the oracle's.  On a
    mismatch, name the first differing position, the keys and payloads found
    and expected there, and what kind of fault it is: keys out of order,
    payloads of equal keys out of input order (a stability fault), or a
    payload that does not travel with its key."""
    got_keys, want_keys = np.asarray(got_keys), np.asarray(want_keys)
    got_vals, want_vals = np.asarray(got_vals), np.asarray(want_vals)
    tag = f"{what}: " if what else ""
    if got_keys.shape != want_keys.shape:
        raise AssertionError(f"{tag}{got_keys.size} keys, expected {want_keys.size}")
    bad = np.flatnonzero(got_keys != want_keys)
    if bad.size:
        i = int(bad[0])
        raise AssertionError(f"{tag}keys differ at {i} of {got_keys.size} ({bad.size} positions): "
                             f"got {int(got_keys[i]):#x}, expected {int(want_keys[i]):#x}")
    if want_vals is None:
        return
    bad = np.flatnonzero(got_vals != want_vals)
    if bad.size:
        i = int(bad[0])
        k = int(got_keys[i])
        tie = np.flatnonzero(want_keys == want_keys[i])
        kind = ("equal keys with payloads out of input order (stability)"
                if int(got_vals[i]) in set(int(v) for v in want_vals[tie]) else
                "a payload that did not travel with its key")
        raise AssertionError(f"{tag}payloads differ at {i} of {got_vals.size} ({bad.size} positions),"
                             f" key {k:#x}: got {int(got_vals[i])}, expected {int(want_vals[i])}: "
                             f"{kind}")
