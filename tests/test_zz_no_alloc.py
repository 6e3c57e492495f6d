"""The key-value sort for callers that cannot allocate device memory.

A caller whose device memory belongs to a pool it may not grow, or a plugin
handed only its input and output buffers, cannot ask for scratch.  The
no-allocation entry point keeps its scratch in a fixed array of the
library's device code instead; it must give exactly what the ordinary entry
point gives (and what the oracle gives), call after call, although every
call reuses (and finds dirty) the same array, and its device-side status
must be readable through its own status call: a look-back wait that runs
out (the probe runs the sort's bounded wait on a word of the array that
nothing sets) is reported there, and the next sort clears it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import poisoned_like, to_dev, to_host

pytestmark = pytest.mark.gpu

MAX_KEYS = 1 << 18


def call_noalloc(lib, dk, dv, ko, vo, n, begin=0, end=32, bits=8):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.radix_sort_pairs_u32_noalloc(
        ctypes.c_void_p(dk.data_ptr()), ctypes.c_void_p(ko.data_ptr()),
        ctypes.c_void_p(dv.data_ptr()), ctypes.c_void_p(vo.data_ptr()),
        n, begin, end, bits, stream)


@pytest.mark.parametrize("n,begin,end,bits", [(100_003, 0, 32, 8), (MAX_KEYS, 0, 32, 4),
                                              (4097, 3, 29, 7)])
def test_no_alloc_matches_ordinary_sort_twice(rs, n, begin, end, bits):
    lib = rs.load_library()
    for call, seed in enumerate((1, 2)):  # two calls in a row, different data
        keys = workloads.u32_uniform(n, seed)
        keys[::5] = keys[0]
        vals = workloads.index_payload(n)
        dk, dv = to_dev(keys), to_dev(vals)
        ko, vo = poisoned_like(dk), poisoned_like(dv)
        assert call_noalloc(lib, dk, dv, ko, vo, n, begin, end, bits) == rs.RS_OK
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert lib.radix_sort_pairs_u32_noalloc_status(stream) == rs.RS_OK
        gk, gv = rs.radix_sort_pairs(dk, dv, begin_bit=begin, end_bit=end, digit_bits=bits)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(ko, np.uint32), to_host(gk, np.uint32)), f"call {call}"
        assert np.array_equal(to_host(vo, np.uint32), to_host(gv, np.uint32)), f"call {call}"
        ek, ev = oracle.sort(keys, vals, begin, end, bits)
        assert np.array_equal(to_host(ko, np.uint32), ek), f"call {call} vs oracle"
        assert np.array_equal(to_host(vo, np.uint32), ev), f"call {call} vs oracle"


def test_no_alloc_rejects_beyond_its_maximum(rs):
    lib = rs.load_library()
    d = torch.empty(4, dtype=torch.int32, device="cuda")
    assert call_noalloc(lib, d, d, d, d, MAX_KEYS + 1) == rs.RS_ERR_INVALID
    assert call_noalloc(lib, d, d, d, d, 0) == rs.RS_OK


def test_no_alloc_status_reports_a_timed_out_wait(rs):
    lib = rs.load_library()
    n = 50_000
    keys, vals = workloads.u32_uniform(n, 9), workloads.index_payload(n)
    dk, dv = to_dev(keys), to_dev(vals)
    ko, vo = poisoned_like(dk), poisoned_like(dv)
    assert call_noalloc(lib, dk, dv, ko, vo, n) == rs.RS_OK  # the array's address is known
    assert rs.noalloc_status() == rs.RS_OK
    assert rs.noalloc_timeout_probe(2_000_000) == rs.RS_ERR_LOOKBACK_TIMEOUT
    assert rs.noalloc_status() == rs.RS_ERR_LOOKBACK_TIMEOUT
    # the next sort starts from a clear status and is right
    ko, vo = poisoned_like(dk), poisoned_like(dv)
    assert call_noalloc(lib, dk, dv, ko, vo, n) == rs.RS_OK
    assert rs.noalloc_status() == rs.RS_OK
    ek, ev = oracle.sort(keys, vals, 0, 32, 8)
    assert np.array_equal(to_host(ko, np.uint32), ek)
    assert np.array_equal(to_host(vo, np.uint32), ev)
