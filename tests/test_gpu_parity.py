"""Parity of the CUDA sort (through the C ABI) with the CPU oracle: bit-exact
keys and payload order, on the workload shapes of the pages and on ragged
and degenerate sizes."""
import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import assert_pairs, field, poisoned_like, to_dev, to_host

pytestmark = pytest.mark.gpu

# tile sizes of the sweep kernels (keys per CTA), so that ragged cases
# straddle tile boundaries
TILE_U32_KEYS, TILE_U32_PAIRS, TILE_U64, TILE_U64_PAIRS, TILE_F16 = 7680, 5888, 5632, 4608, 6144
# flat u32 sorts of at most MID_MAX keys use the smaller mid-size tiles
MID_KEYS, MID_PAIRS, MID_MAX = 3584, 3072, 1 << 18


def run_keys(rs, keys, begin=0, end=None, bits=8, **opts):
    d = to_dev(keys)
    out = poisoned_like(d)
    rs.radix_sort_keys(d, out, begin, end, bits, **opts)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(d, keys.dtype), keys), "input was written"
    return to_host(out, keys.dtype)


def run_pairs(rs, keys, vals, begin=0, end=None, bits=8, **opts):
    dk, dv = to_dev(keys), to_dev(vals)
    ko, vo = poisoned_like(dk), poisoned_like(dv)
    rs.radix_sort_pairs(dk, dv, ko, vo, begin, end, bits, **opts)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(dk, keys.dtype), keys), "input keys were written"
    assert np.array_equal(to_host(dv, vals.dtype), vals), "input payloads were written"
    return to_host(ko, keys.dtype), to_host(vo, vals.dtype)


# ------------------------------------------------------------ page workloads

def test_1024_keys_below_4096_three_hex_passes(rs):
    keys = workloads.u32_small(1024, 0, 12)
    got = run_keys(rs, keys, 0, 12, 4)
    exp, _ = oracle.sort(keys, None, 0, 12, 4)
    assert np.array_equal(got, exp)
    kp, vp = run_pairs(rs, keys, workloads.index_payload(1024), 0, 12, 4)
    ek, ev = oracle.sort(keys, workloads.index_payload(1024), 0, 12, 4)
    assert_pairs(kp, vp, ek, ev)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("bits", [4, 8])
def test_4m_uniform_keys(rs, seed, bits):
    keys = workloads.u32_uniform(4_194_304, seed)
    got = run_keys(rs, keys, 0, 32, bits)
    exp, _ = oracle.sort(keys, None, 0, 32, bits)
    assert np.array_equal(got, exp)


def test_page_size_not_a_tile_multiple(rs):
    # 4,194,915 keys: the day-35 page's count, not a multiple of any tile
    keys = workloads.u32_uniform(4_194_915, 5)
    vals = workloads.index_payload(keys.size)
    for bits in (4, 8):
        ko, vo = run_pairs(rs, keys, vals, 0, 32, bits)
        ek, ev = oracle.sort(keys, vals, 0, 32, bits)
        assert_pairs(ko, vo, ek, ev)


@pytest.mark.parametrize("dist", list(workloads.U32_DISTRIBUTIONS))
def test_pairs_distributions(rs, dist):
    n = 3 * (1 << 20) + 12345
    keys = workloads.U32_DISTRIBUTIONS[dist](n, 0)
    vals = workloads.index_payload(n)
    ko, vo = run_pairs(rs, keys, vals, 0, 32, 8)
    ek, ev = oracle.sort(keys, vals, 0, 32, 8)
    assert np.array_equal(ko, ek)
    assert np.array_equal(vo, ev)


@pytest.mark.parametrize("dist", list(workloads.U64_DISTRIBUTIONS))
@pytest.mark.parametrize("begin,end", [(0, 64), (0, 40), (13, 57)])
def test_u64_pairs_and_keys(rs, dist, begin, end):
    n = (1 << 21) + 77
    keys = workloads.U64_DISTRIBUTIONS[dist](n, 0)
    vals = workloads.index_payload(n)
    ko, vo = run_pairs(rs, keys, vals, begin, end, 8)
    ek, ev = oracle.sort(keys, vals, begin, end, 8)
    assert_pairs(ko, vo, ek, ev)
    k2 = run_keys(rs, keys, begin, end, 8)
    assert np.array_equal(k2, ek)


# ---------------------------------------------------- ragged and degenerate

RAGGED = [1, 2, 31, 32, 33, 1000, TILE_U64 - 1, TILE_U64, TILE_U64 + 1, TILE_U64_PAIRS - 1,
          TILE_U64_PAIRS + 1, MID_PAIRS - 1, MID_PAIRS + 1, MID_KEYS - 1, MID_KEYS,
          MID_KEYS + 1, 3 * MID_KEYS + 17, 100_003]


@pytest.mark.parametrize("n", RAGGED)
@pytest.mark.parametrize("small_sort", [True, False], ids=["one_kernel_short_rows",
                                                          "multi_kernel_only"])
def test_ragged_sizes(rs, n, small_sort):
    # Inputs of at most rs.SMALL_SORT_MAX_KEYS keys are sorted by one kernel;
    # with small_sort=False the tile-boundary sizes exercise the scatter
    # kernels (full and partial tiles) instead.
    o = {"small_sort": small_sort}
    keys = workloads.u32_uniform(n, 11)
    keys[::3] = keys[0]  # ties across tiles
    vals = workloads.index_payload(n)
    for bits in (8, 5):
        ko, vo = run_pairs(rs, keys, vals, 0, 32, bits, **o)
        ek, ev = oracle.sort(keys, vals, 0, 32, bits)
        assert_pairs(ko, vo, ek, ev, f"b={bits}")
        assert np.array_equal(run_keys(rs, keys, 0, 32, bits, **o), ek)
    k64 = workloads.u64_uniform(n, 12)
    assert np.array_equal(run_keys(rs, k64, 0, 64, 8, **o), oracle.sort(k64, None, 0, 64, 8)[0])
    k64o, v64o = run_pairs(rs, k64, vals, 0, 64, 8, **o)
    e64, ev64 = oracle.sort(k64, vals, 0, 64, 8)
    assert_pairs(k64o, v64o, e64, ev64)


@pytest.mark.parametrize("n", [MID_MAX, MID_MAX + 1, 36 * TILE_U32_KEYS, 36 * TILE_U32_KEYS + 1,
                               45 * TILE_U32_PAIRS - 1, 45 * TILE_U32_PAIRS + 1])
def test_tile_shapes_either_side_of_mid_size(rs, n):
    # up to MID_MAX keys the mid-size tiles, above it the large ones, with
    # full and partial last tiles of each
    keys = workloads.u32_uniform(n, 31)
    keys[::4] = keys[1]
    vals = workloads.index_payload(n)
    ko, vo = run_pairs(rs, keys, vals, 0, 32, 8)
    ek, ev = oracle.sort(keys, vals, 0, 32, 8)
    assert_pairs(ko, vo, ek, ev)
    assert np.array_equal(run_keys(rs, keys, 0, 32, 8), ek)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_digit_width(rs, bits):
    n = 50_001
    keys = (workloads.words(21, 0, n) >> np.uint64(40)).astype(np.uint32)  # 24-bit keys
    vals = workloads.index_payload(n)
    ko, vo = run_pairs(rs, keys, vals, 0, 24, bits)
    ek, ev = oracle.sort(keys, vals, 0, 24, bits)
    assert_pairs(ko, vo, ek, ev)
    k64 = workloads.u64_uniform(n, 22)
    k64o, v64o = run_pairs(rs, k64, vals, 5, 37, bits)
    e64, ev64 = oracle.sort(k64, vals, 5, 37, bits)
    assert_pairs(k64o, v64o, e64, ev64)


@pytest.mark.parametrize("begin,end,bits", [(0, 1, 1), (31, 32, 8), (3, 29, 7), (8, 24, 3),
                                            (0, 12, 4), (16, 32, 8)])
def test_bit_ranges(rs, begin, end, bits):
    n = 70_000
    keys = workloads.u32_uniform(n, 3)
    vals = workloads.index_payload(n)
    ko, vo = run_pairs(rs, keys, vals, begin, end, bits)
    ek, ev = oracle.sort(keys, vals, begin, end, bits)
    assert_pairs(ko, vo, ek, ev, f"bits [{begin}, {end}) b={bits}")


def test_one_key_and_all_equal_small(rs):
    for n in (1, 7, 8192 * 2 + 1):
        keys = np.full(n, 0xDEADBEEF, np.uint32)
        vals = workloads.index_payload(n)
        ko, vo = run_pairs(rs, keys, vals)
        ek, ev = oracle.sort(keys, vals, 0, 32, 8)
        assert_pairs(ko, vo, ek, ev, f"n={n}")


def test_empty_input(rs):
    d = torch.empty(0, dtype=torch.int32, device="cuda")
    out = rs.radix_sort_keys(d)
    assert out.numel() == 0


@pytest.mark.parametrize("bits,end", [(8, 32), (8, 24), (4, 32)])
def test_in_place(rs, bits, end):
    # even (4 or 8) and odd (3) pass counts; odd ones end with one copy
    n = 123_457
    keys = workloads.u32_uniform(n, 9)
    vals = workloads.index_payload(n)
    dk, dv = to_dev(keys), to_dev(vals)
    rs.radix_sort_pairs(dk, dv, dk, dv, 0, end, bits)
    ek, ev = oracle.sort(keys, vals, 0, end, bits)
    assert np.array_equal(to_host(dk, np.uint32), ek)
    assert np.array_equal(to_host(dv, np.uint32), ev)


def test_max_digit_runs_cross_many_tiles(rs):
    # two digits alternate in long runs: every tile holds one or two digits
    n = 40 * TILE_U32_PAIRS + 3
    keys = np.repeat(np.array([0x01000000, 0x00000001], np.uint32), n // 2 + 1)[:n].copy()
    keys[::2] ^= np.uint32(0x00010000)
    vals = workloads.index_payload(n)
    ko, vo = run_pairs(rs, keys, vals)
    ek, ev = oracle.sort(keys, vals)
    assert_pairs(ko, vo, ek, ev)


# -------------------------------------------------------------- histograms

@pytest.mark.parametrize("dtype,begin,end,bits", [(np.uint32, 0, 32, 8), (np.uint32, 0, 32, 4),
                                                  (np.uint64, 0, 64, 8), (np.uint64, 0, 40, 8),
                                                  (np.uint32, 5, 30, 6)])
def test_upfront_histograms_and_scan(rs, dtype, begin, end, bits):
    n = (1 << 22) + 999
    keys = workloads.words(4, 0, n)
    if dtype == np.uint32:
        keys = (keys >> np.uint64(32)).astype(np.uint32)
    hist, bases = rs.upfront_histograms(to_dev(keys), begin, end, bits)
    hist = to_host(hist, np.uint32).astype(np.uint64)
    bases = to_host(bases, np.uint32).astype(np.uint64)
    exp = oracle.pass_histograms(keys, begin, end, bits)
    assert np.array_equal(hist, exp)
    excl = np.concatenate([np.zeros((exp.shape[0], 1), np.uint64),
                           np.cumsum(exp, axis=1)[:, :-1]], axis=1)
    assert np.array_equal(bases, excl)


def test_upfront_histograms_skewed(rs):
    for keys in (workloads.u32_all_equal(1 << 20), workloads.u32_low_entropy(1 << 20)):
        hist, _ = rs.upfront_histograms(to_dev(keys))
        assert np.array_equal(to_host(hist, np.uint32).astype(np.uint64),
                              oracle.pass_histograms(keys))


# ------------------------------------------------------------ row-wise sort

@pytest.mark.parametrize("kind", ["f16", "bf16"])
@pytest.mark.parametrize("descending", [False, True])
def test_segmented_page_shape(rs, kind, descending):
    x = workloads.rows16(1024, 65536, kind, seed=0)
    dt = torch.float16 if kind == "f16" else torch.bfloat16
    d = to_dev(x).view(dt)
    vals, idx = rs.segmented_sort(d, descending)
    torch.cuda.synchronize()
    ev, ei = oracle.segmented_sort16(x, descending)
    assert np.array_equal(to_host(vals.view(torch.int16), np.uint16), ev)
    assert np.array_equal(idx.cpu().numpy(), ei)
    assert np.array_equal(to_host(d.view(torch.int16), np.uint16), x), "input was written"


@pytest.mark.parametrize("shape", [(1, 1), (3, 1000), (64, 64), (7, 4097), (3, 8192), (3, 8193),
                                   (2, 2 * TILE_F16), (2, 2 * TILE_F16 + 1),
                                   (3, 3 * TILE_F16 - 1), (2, 200_001),
                                   (16, 131072), (1024, 1), (5, 0), (0, 7)])
@pytest.mark.parametrize("descending", [False, True])
def test_segmented_shapes(rs, shape, descending):
    rows, cols = shape
    x = workloads.rows16(rows, cols, "f16", seed=3)
    d = to_dev(x).view(torch.float16)
    vals, idx = rs.segmented_sort(d, descending)
    torch.cuda.synchronize()
    ev, ei = oracle.segmented_sort16(x, descending)
    assert np.array_equal(to_host(vals.view(torch.int16), np.uint16), ev)
    assert np.array_equal(idx.cpu().numpy(), ei)


def test_segmented_matches_torch_sort_on_finite_rows(rs):
    """Informational cross-check: without NaNs and signed zeros the order is
    torch.sort's (stable) order."""
    x = workloads.rows16(8, 10_000, "bf16", seed=4)
    bad = (x == 0x8000) | ((x & 0x7F80) == 0x7F80) & ((x & 0x7F) != 0)
    x[bad] = 0x3F80
    d = to_dev(x).view(torch.bfloat16)
    vals, idx = rs.segmented_sort(d, False)
    tv, ti = torch.sort(d, dim=-1, stable=True)
    assert torch.equal(idx, ti)
    assert torch.equal(vals.view(torch.int16), tv.view(torch.int16))


# ------------------------------------------------------- failure detection

def test_lookback_wait_times_out_on_unset_word(rs):
    # the wait runs on a word that nothing sets; it must give up and report
    status = rs.lookback_timeout_probe(2_000_000)  # 2 ms
    assert status == rs.RS_ERR_LOOKBACK_TIMEOUT
    # the context is still usable and a normal sort reports no device error
    keys = workloads.u32_uniform(100_000, 1)
    d = to_dev(keys)
    temp = torch.empty(rs.temp_bytes(keys.size, 4, 0, 0, 32, 8), dtype=torch.uint8, device="cuda")
    out = rs.radix_sort_keys(d, temp=temp)
    assert rs.device_status(temp) == rs.RS_OK
    assert np.array_equal(to_host(out, np.uint32), np.sort(keys))


def test_copy_probe(rs):
    src = torch.randint(0, 2**31 - 1, (1 << 22,), dtype=torch.int32, device="cuda")
    dst = torch.zeros_like(src)
    rs.copy_probe(dst, src)
    assert torch.equal(src, dst)
