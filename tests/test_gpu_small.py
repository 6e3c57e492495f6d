"""Sorts of at most 8,192 keys per row run in one kernel (every pass in one
CTA's shared memory): parity with the oracle at and around the three small
tile sizes, for every key kind, both payload kinds, 4- and 8-bit digits,
partial bit ranges, in place, and rows."""
import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import poisoned_like, to_dev, to_host
from tests.test_gpu_typed import same_bits, typed_keys

pytestmark = pytest.mark.gpu

SMALL = [1, 2, 31, 32, 33, 255, 1023, 1024, 1025, 2049, 4095, 4096, 4097, 6001, 8191, 8192]


@pytest.mark.parametrize("n", SMALL)
@pytest.mark.parametrize("bits", [4, 8])
def test_small_u32_u64(rs, n, bits):
    keys = workloads.u32_uniform(n, n)
    keys[::4] = keys[0]
    vals = workloads.index_payload(n)
    dk, dv = to_dev(keys), to_dev(vals)
    ko, vo = poisoned_like(dk), poisoned_like(dv)
    rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, bits)
    ek, ev = oracle.sort(keys, vals, 0, 32, bits)
    assert np.array_equal(to_host(ko, np.uint32), ek) and np.array_equal(to_host(vo, np.uint32), ev)
    k64 = workloads.u64_uniform(n, n + 1)
    d64 = to_dev(k64)
    o64 = poisoned_like(d64)
    rs.radix_sort_keys(d64, o64, 3, 61, bits)
    assert np.array_equal(to_host(o64, np.uint64), oracle.sort(k64, None, 3, 61, bits)[0])


@pytest.mark.parametrize("key_type", ["i32", "f32", "i64", "f64"])
@pytest.mark.parametrize("n", [7, 1024, 3001, 7777])
def test_small_typed(rs, key_type, n):
    keys = typed_keys(key_type, n, 90 + n)
    vals = workloads.index_payload(n)
    for descending in (False, True):
        dk, dv = to_dev(keys), to_dev(vals)
        ko, vo = poisoned_like(dk), poisoned_like(dv)
        rs.radix_sort_pairs(dk, dv, ko, vo, key_type=key_type, descending=descending)
        ek, ev = oracle.sort_typed(keys, key_type, vals, descending)
        assert same_bits(to_host(ko, keys.dtype), ek) and np.array_equal(to_host(vo, np.uint32), ev)


def test_small_in_place(rs):
    n = 3000
    keys = workloads.u32_uniform(n, 5)
    vals = workloads.index_payload(n)
    dk, dv = to_dev(keys), to_dev(vals)
    rs.radix_sort_pairs(dk, dv, dk, dv, 0, 32, 8)
    ek, ev = oracle.sort(keys, vals, 0, 32, 8)
    assert np.array_equal(to_host(dk, np.uint32), ek) and np.array_equal(to_host(dv, np.uint32), ev)


@pytest.mark.parametrize("shape", [(1, 1), (3, 17), (100, 1024), (7, 4096), (2, 4095), (5, 4097),
                                   (3, 8192), (200, 6000)])
def test_small_rows(rs, shape):
    h = workloads.rows16(*shape, "f16", seed=shape[1])
    x = torch.from_numpy(h.view(np.int16)).cuda().view(torch.float16)
    for descending in (False, True):
        v, i = rs.segmented_sort(x, descending)
        ev, ei = oracle.segmented_sort16(h, descending)
        assert np.array_equal(v.view(torch.int16).cpu().numpy().view(np.uint16), ev)
        assert np.array_equal(i.cpu().numpy(), ei)


def test_small_sort_switch(rs):
    """With the one-kernel path off, the same short inputs take the
    multi-kernel path and give the same results."""
    n = 6001
    keys = workloads.u32_uniform(n, 17)
    vals = workloads.index_payload(n)
    ek, ev = oracle.sort(keys, vals, 0, 32, 8)
    for on in (False, True):
        dk, dv = to_dev(keys), to_dev(vals)
        ko, vo = poisoned_like(dk), poisoned_like(dv)
        rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, 8, small_sort=on)
        assert np.array_equal(to_host(ko, np.uint32), ek)
        assert np.array_equal(to_host(vo, np.uint32), ev)
