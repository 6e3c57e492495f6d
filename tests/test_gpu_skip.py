"""Passes in which every key has the same digit are the identity and are
skipped on the device (the schedule comes from the upfront histograms).
Parity with the oracle, and the number of passes run, for sorts with
0, 1, 3 and 5 of their passes run, in and out of place, for keys, pairs,
typed keys and row-wise 16-bit sorts.  Pass skipping is an option of each
call (pass_skipping=True), never a state of the library."""
import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import assert_pairs, poisoned_like, to_dev, to_host

pytestmark = pytest.mark.gpu


def sort_pairs(rs, keys, vals, begin, end, bits, in_place, skip=True, **kw):
    dk, dv = to_dev(keys), to_dev(vals)
    kb = keys.dtype.itemsize
    temp = torch.empty(rs.temp_bytes(keys.size, kb, 4, begin, end, bits), dtype=torch.uint8,
                       device="cuda")
    if in_place:
        rs.radix_sort_pairs(dk, dv, dk, dv, begin, end, bits, temp=temp, pass_skipping=skip,
                            **kw)
        ko, vo = dk, dv
    else:
        ko, vo = poisoned_like(dk), poisoned_like(dv)
        rs.radix_sort_pairs(dk, dv, ko, vo, begin, end, bits, temp=temp, pass_skipping=skip,
                            **kw)
    run = rs.passes_run(temp)
    return to_host(ko, keys.dtype), to_host(vo, vals.dtype), run


def sort_keys(rs, keys, begin, end, bits, in_place, **kw):
    dk = to_dev(keys)
    kb = keys.dtype.itemsize
    temp = torch.empty(rs.temp_bytes(keys.size, kb, 0, begin, end, bits), dtype=torch.uint8,
                       device="cuda")
    ko = dk if in_place else poisoned_like(dk)
    rs.radix_sort_keys(dk, ko, begin, end, bits, temp=temp, pass_skipping=True, **kw)
    return to_host(ko, keys.dtype), rs.passes_run(temp)


CASES = {
    # u64 keys below 2^40, all 64 bits sorted: the top three 8-bit passes skip
    "u64_40bit": (lambda n: workloads.u64_uniform(n, 3) & np.uint64((1 << 40) - 1), 0, 64, 8, 5),
    # u32 keys whose bits 8..15 are constant: one of four passes skips
    "u32_const_byte": (lambda n: (workloads.u32_uniform(n, 4) & np.uint32(0xFFFF00FF))
                       | np.uint32(0x5A00), 0, 32, 8, 3),
    # every key equal: no pass runs, the input is copied
    "all_equal": (lambda n: np.full(n, 0xDEADBEEF, np.uint32), 0, 32, 8, 0),
    # one 4-bit digit of six varies: one pass runs
    "u32_one_digit": (lambda n: (workloads.u32_uniform(n, 5) & np.uint32(0x00000F00))
                      | np.uint32(0x7000000), 0, 24, 4, 1),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("n", [1000, 5889, 9001, 300_001])
def test_skipped_passes_pairs(rs, case, in_place, n):
    make, begin, end, bits, want_run = CASES[case]
    keys = make(n)
    vals = workloads.index_payload(n)
    ek, ev = oracle.sort(keys, vals, begin, end, bits)
    ko, vo, run = sort_pairs(rs, keys, vals, begin, end, bits, in_place)
    assert_pairs(ko, vo, ek, ev)
    # short inputs are sorted by one kernel in shared memory, every pass
    # included
    assert run == (want_run if n > rs.SMALL_SORT_MAX_KEYS else oracle.num_passes(begin, end, bits))


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("in_place", [False, True])
def test_skipped_passes_keys(rs, case, in_place):
    make, begin, end, bits, want_run = CASES[case]
    keys = make(77_777)
    ek, _ = oracle.sort(keys, None, begin, end, bits)
    ko, run = sort_keys(rs, keys, begin, end, bits, in_place)
    assert np.array_equal(ko, ek)
    assert run == want_run


def test_skipping_off_runs_every_pass(rs):
    make, begin, end, bits, _ = CASES["u32_const_byte"]
    keys = make(50_001)
    vals = workloads.index_payload(50_001)
    ek, ev = oracle.sort(keys, vals, begin, end, bits)
    for in_place in (False, True):
        ko, vo, run = sort_pairs(rs, keys, vals, begin, end, bits, in_place, skip=False)
        assert_pairs(ko, vo, ek, ev)
        assert run == 4


def test_no_pass_skipped_on_uniform_keys(rs):
    keys = workloads.u32_uniform(100_000, 6)
    vals = workloads.index_payload(100_000)
    ko, vo, run = sort_pairs(rs, keys, vals, 0, 32, 8, False)
    ek, ev = oracle.sort(keys, vals, 0, 32, 8)
    assert_pairs(ko, vo, ek, ev)
    assert run == 4


@pytest.mark.parametrize("in_place", [False, True])
def test_typed_skips_on_transformed_digits(rs, in_place):
    # floats in [1, 2): the top byte of the transformed key is constant
    n = 60_000
    x = (1.0 + (workloads.u32_uniform(n, 7) >> np.uint32(9)).astype(np.float64) / 2.0**23)
    x = x.astype(np.float32)
    vals = workloads.index_payload(n)
    for descending in (False, True):
        ek, ev = oracle.sort_typed(x, "f32", vals, descending)
        ko, vo, run = sort_pairs(rs, x, vals, 0, 32, 8, in_place, key_type="f32",
                                 descending=descending)
        assert np.array_equal(ko.view(np.uint32), ek.view(np.uint32))
        assert np.array_equal(vo, ev) and run == 3


# Signed, float and descending keys carry T(k) between the first and the
# last pass run: one pass run (first and last at once), none (the input is
# copied), an even and an odd number in place, for 32- and 64-bit keys.
TYPED_CASES = {
    "i32_one_byte": (lambda n: (workloads.u32_uniform(n, 11) & np.uint32(0xFF)).astype(np.int32),
                     "i32", 1),
    "i32_all_equal": (lambda n: np.full(n, -12345, np.int32), "i32", 0),
    "i64_two_bytes": (lambda n: (workloads.u64_uniform(n, 12) & np.uint64(0xFFFF)).astype(np.int64),
                      "i64", 2),
    "f64_seven_bytes": (lambda n: 1.0 + (workloads.u64_uniform(n, 13) >> np.uint64(12)).astype(
        np.float64) / 2.0**52, "f64", 7),
}


@pytest.mark.parametrize("case", sorted(TYPED_CASES))
@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("descending", [False, True])
def test_typed_passes_run_carry_the_transform(rs, case, in_place, descending):
    gen, key_type, want = TYPED_CASES[case]
    n = 40_001
    x = gen(n)
    vals = workloads.index_payload(n)
    ek, ev = oracle.sort_typed(x, key_type, vals, descending)
    end = 8 * x.dtype.itemsize
    ko, vo, run = sort_pairs(rs, x, vals, 0, end, 8, in_place, key_type=key_type,
                             descending=descending)
    u = np.uint32 if x.dtype.itemsize == 4 else np.uint64
    assert np.array_equal(ko.view(u), ek.view(u))
    assert np.array_equal(vo, ev) and run == want


def _rows_sort(rs, x, descending, in_place=False):
    d = torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)
    temp = torch.empty(rs.segmented_temp_bytes(*x.shape), dtype=torch.uint8, device="cuda")
    vals = d if in_place else None
    v, i = rs.segmented_sort(d, descending, values_out=vals, temp=temp, pass_skipping=True)
    return v.view(torch.int16).cpu().numpy().view(np.uint16), i.cpu().numpy(), rs.passes_run(temp)


@pytest.mark.parametrize("descending", [False, True])
@pytest.mark.parametrize("in_place", [False, True])
def test_rows_skip(rs, descending, in_place):
    rows, cols = 6, 10_000
    w = workloads.words(8, 0, rows * cols).reshape(rows, cols)
    # every row: patterns 0x3C00..0x3CFF (one high byte): the second pass skips
    one_byte = (np.uint64(0x3C00) | (w & np.uint64(0xFF))).astype(np.uint16)
    # every row constant: no pass runs, the indices are the identity
    const = np.full((rows, cols), 0x4248, np.uint16)
    # only one row with one high byte: no pass skips
    mixed = (w & np.uint64(0xFFFF)).astype(np.uint16)
    mixed[2] = one_byte[2]
    for x, want_run in ((one_byte, 1), (const, 0), (mixed, 2)):
        ev, ei = oracle.segmented_sort16(x, descending)
        v, i, run = _rows_sort(rs, x.copy(), descending, in_place)
        assert np.array_equal(v, ev) and np.array_equal(i, ei)
        assert run == want_run
