"""Parity of the typed global sorts (signed and IEEE float keys, ascending
and descending, through radix_sort_keys_typed / radix_sort_pairs_typed)
with the oracle: bit-exact keys and payload order, on ragged sizes, special
values, narrower digits and bit ranges of the transformed key."""
import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import poisoned_like, to_dev, to_host

pytestmark = pytest.mark.gpu

TILE_32_KEYS, TILE_32_PAIRS, TILE_64_KEYS, TILE_64_PAIRS = 7680, 5888, 5632, 4608
SIZES = [1, 2, 33, 1000, TILE_32_PAIRS - 1, TILE_32_PAIRS + 1, TILE_32_KEYS + 1,
         TILE_64_PAIRS + 1, 3 * TILE_32_KEYS + 17, 100_003]
TYPES = {"i32": np.int32, "f32": np.float32, "i64": np.int64, "f64": np.float64,
         "u32": np.uint32, "u64": np.uint64}
F32_SPECIAL = np.array([0xFFC00000, 0xFF800000, 0xFF7FFFFF, 0xBF800000, 0x80000001, 0x80000000,
                        0x00000000, 0x00000001, 0x3F800000, 0x7F7FFFFF, 0x7F800000, 0x7FC00000],
                       np.uint32)
F64_SPECIAL = np.array([0xFFF8000000000000, 0xFFF0000000000000, 0xFFEFFFFFFFFFFFFF,
                        0xBFF0000000000000, 0x8000000000000001, 0x8000000000000000, 0,
                        1, 0x3FF0000000000000, 0x7FEFFFFFFFFFFFFF, 0x7FF0000000000000,
                        0x7FF8000000000000], np.uint64)


def typed_keys(key_type: str, n: int, seed: int) -> np.ndarray:
    """Seeded keys of a type: uniform bit patterns mixed with ties, both
    zeros, infinities, NaNs of both signs and subnormals (floats)."""
    dt = TYPES[key_type]
    size = np.dtype(dt).itemsize
    w = workloads.words(seed, 30, n)
    bits = (w >> np.uint64(32)).astype(np.uint32) if size == 4 else w.copy()
    if key_type.startswith("f"):
        # mostly finite values of moderate magnitude, plus special patterns
        x = ((w >> np.uint64(11)).astype(np.float64) / 2.0**53 - 0.5) * 2e4
        bits = x.astype(dt).view(bits.dtype)
        special = F32_SPECIAL if size == 4 else F64_SPECIAL
        pick = workloads.words(seed, 31, n) % np.uint64(16)
        sel = pick < np.uint64(len(special))
        bits[sel] = special[pick[sel].astype(np.int64)]
    bits[::9] = bits[min(4, n - 1)]  # ties
    return bits.view(dt)


def run_typed(rs, keys, key_type, descending, vals=None, begin=0, end=None, bits=8):
    dk = to_dev(keys)
    ko = poisoned_like(dk)
    if vals is None:
        rs.radix_sort_keys(dk, ko, begin, end, bits, key_type=key_type, descending=descending)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(dk, keys.dtype).view(np.uint8), keys.view(np.uint8))
        return to_host(ko, keys.dtype), None
    dv = to_dev(vals)
    vo = poisoned_like(dv)
    rs.radix_sort_pairs(dk, dv, ko, vo, begin, end, bits, key_type=key_type,
                        descending=descending)
    torch.cuda.synchronize()
    return to_host(ko, keys.dtype), to_host(vo, vals.dtype)


def same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8),
                          np.ascontiguousarray(b).view(np.uint8))


@pytest.mark.parametrize("key_type", ["i32", "f32", "i64", "f64"])
@pytest.mark.parametrize("descending", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_typed_keys_and_pairs(rs, key_type, descending, n):
    keys = typed_keys(key_type, n, 40 + n % 7)
    vals = workloads.index_payload(n)
    ek, ev = oracle.sort_typed(keys, key_type, vals, descending)
    ko, _ = run_typed(rs, keys, key_type, descending)
    assert same_bits(ko, ek)
    kp, vp = run_typed(rs, keys, key_type, descending, vals)
    assert same_bits(kp, ek) and np.array_equal(vp, ev)


@pytest.mark.parametrize("key_type", ["u32", "u64"])
def test_unsigned_descending(rs, key_type):
    n = 70_001
    keys = typed_keys(key_type, n, 50)
    vals = workloads.index_payload(n)
    ek, ev = oracle.sort_typed(keys, key_type, vals, True)
    kp, vp = run_typed(rs, keys, key_type, True, vals)
    assert same_bits(kp, ek) and np.array_equal(vp, ev)


@pytest.mark.parametrize("key_type", ["i32", "f32", "f64"])
@pytest.mark.parametrize("bits", [1, 3, 5, 7])
def test_typed_digit_widths(rs, key_type, bits):
    n = 30_011
    keys = typed_keys(key_type, n, 60 + bits)
    vals = workloads.index_payload(n)
    for descending in (False, True):
        ek, ev = oracle.sort_typed(keys, key_type, vals, descending, digit_bits=bits)
        kp, vp = run_typed(rs, keys, key_type, descending, vals, bits=bits)
        assert same_bits(kp, ek) and np.array_equal(vp, ev)


@pytest.mark.parametrize("key_type,begin,end", [("i32", 8, 24), ("f32", 20, 32), ("i64", 3, 40),
                                                ("f64", 52, 64)])
def test_typed_bit_ranges(rs, key_type, begin, end):
    n = 50_000
    keys = typed_keys(key_type, n, 70)
    vals = workloads.index_payload(n)
    for descending in (False, True):
        ek, ev = oracle.sort_typed(keys, key_type, vals, descending, begin, end, 8)
        kp, vp = run_typed(rs, keys, key_type, descending, vals, begin, end, 8)
        assert same_bits(kp, ek) and np.array_equal(vp, ev)


def test_special_values_order(rs):
    # every special pattern, many times, in a shuffled order
    reps = 500
    for special, dt, key_type in ((F32_SPECIAL, np.float32, "f32"), (F64_SPECIAL, np.float64, "f64")):
        idx = (workloads.words(80, 0, reps * len(special)) % np.uint64(len(special))).astype(np.int64)
        keys = special[idx].view(dt)
        for descending in (False, True):
            ko, _ = run_typed(rs, keys, key_type, descending)
            want = np.sort(idx)[::-1] if descending else np.sort(idx)
            assert same_bits(ko, special[want].view(dt))


def test_typed_key_type_must_match_the_tensor(rs):
    with pytest.raises(TypeError):
        rs.radix_sort_keys(torch.zeros(4, dtype=torch.float32, device="cuda"), key_type="f64")
