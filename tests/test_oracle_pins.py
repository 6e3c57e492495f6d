"""Pins for the CPU oracle: it is checked against things other than itself.

* values the pages print for worked examples (tests/golden/);
* the closed form of a stable sort's destination,
      pos(i) = #{j : f(k_j) < f(k_i)} + #{j < i : f(k_j) = f(k_i)},
  evaluated by brute force for every short input;
* numpy's stable argsort as a library special case;
* invariants: permutation, non-decreasing sort field, ties in input order;
* the float order of every 16-bit pattern for the order-preserving bijection.
"""
import itertools

import numpy as np
import pytest

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.conftest import read_golden


def rank_positions(f):
    """Closed-form stable destination of every element (O(n^2))."""
    f = np.asarray(f, dtype=np.int64)
    less = (f[None, :] < f[:, None]).sum(axis=1)
    eq_before = np.tril(f[None, :] == f[:, None], -1).sum(axis=1)
    return less + eq_before


def field(keys, begin, end):
    keys = np.asarray(keys).astype(np.uint64)
    w = end - begin
    mask = np.uint64((1 << w) - 1) if w < 64 else np.uint64(0xFFFFFFFFFFFFFFFF)
    return (keys >> np.uint64(begin)) & mask


# ------------------------------------------------------------- worked examples

def test_base10_histogram_and_offsets():
    g = read_golden("base10_worked_example.txt")
    a = np.array(g["input"])
    base = g["base"][0]
    digits = (a // 1) % base
    assert digits.tolist() == g["place1_digits"]
    counts, offsets, dest = oracle.counting_pass(digits, base)
    assert counts.tolist() == g["place1_counts"]
    assert offsets.tolist() == g["place1_offsets"]
    assert int(counts.sum()) == len(a)


def test_base10_one_stable_pass():
    g = read_golden("base10_worked_example.txt")
    a = np.array(g["input"])
    digits = a % 10
    counts, offsets, dest = oracle.counting_pass(digits, 10)
    out = np.empty_like(a)
    idx = np.empty_like(a)
    out[dest.astype(np.int64)] = a
    idx[dest.astype(np.int64)] = np.arange(len(a))
    assert out.tolist() == g["pass1_values"]
    assert idx.tolist() == g["pass1_indices"]
    rank = dest.astype(np.int64) - offsets[digits].astype(np.int64)
    assert rank.tolist() == g["place1_rank_within_digit"]
    # digit 3's indicator and its exclusive scan are the ranks of its members
    ind = (digits == 3).astype(np.int64)
    assert ind.tolist() == g["digit3_indicator"]
    excl = np.concatenate([[0], np.cumsum(ind)[:-1]])
    assert excl.tolist() == g["digit3_exclusive_scan"]
    assert rank[digits == 3].tolist() == excl[digits == 3].tolist()
    # the two 13s (indices 1 and 6) keep their input order
    assert [i for i in idx.tolist() if a[i] == 13] == [1, 6]


def test_base10_two_passes():
    g = read_golden("base10_worked_example.txt")
    a = np.array(g["input"])
    idx = np.arange(len(a))
    place = 1
    while place <= a.max():
        _, _, dest = oracle.counting_pass((a // place) % 10, 10)
        d = dest.astype(np.int64)
        na, ni = np.empty_like(a), np.empty_like(idx)
        na[d], ni[d] = a, idx
        a, idx = na, ni
        place *= 10
    assert place == 100  # two passes for a two-digit maximum
    assert a.tolist() == g["pass2_values"]
    assert idx.tolist() == g["pass2_indices"]


def test_one_bit_split_16_keys():
    g = read_golden("one_bit_split_16.txt")
    keys = np.array(g["keys"], np.uint32)
    clear = g["clear_count"][0]
    flag = 1 - (keys & 1).astype(np.int64)               # 1 marks a clear key
    f = np.concatenate([[0], np.cumsum(flag)[:-1]])      # exclusive scan
    total_falses = f[-1] + flag[-1]
    assert total_falses == clear == 9
    i = np.arange(16)
    dst = np.where(keys & 1, total_falses + i - f, f)
    assert sorted(dst.tolist()) == list(range(16))
    # the oracle's one-bit pass puts every key at the page's destination
    kout, vout = oracle.sort(keys, np.arange(16, dtype=np.uint32), 0, 1, 1)
    expect = np.empty(16, np.uint32)
    expect[dst] = keys
    assert kout.tolist() == expect.tolist()
    assert vout[:9].tolist() == np.nonzero(flag)[0].tolist()
    assert vout[9:].tolist() == np.nonzero(1 - flag)[0].tolist()


def test_1024_keys_below_4096_three_hex_passes():
    keys = workloads.u32_small(1024, seed=0, bits=12)
    assert keys.max() < 4096
    assert oracle.num_passes(0, 12, 4) == 3
    kout, vout = oracle.sort(keys, workloads.index_payload(1024), 0, 12, 4)
    pos = rank_positions(keys)
    expect = np.empty_like(keys)
    expect[pos] = keys
    assert kout.tolist() == expect.tolist()
    eidx = np.empty(1024, np.int64)
    eidx[pos] = np.arange(1024)
    assert vout.tolist() == eidx.tolist()
    print("first/middle/last:", kout[0], kout[511], kout[-1])


# ----------------------------------------------------------------- brute force

@pytest.mark.parametrize("b", [1, 2, 3])
def test_brute_force_all_short_inputs(b):
    """Every array of length <= 5 over 3-bit keys (and a seeded sample of
    length-6 arrays) against the closed-form stable positions."""
    cases = []
    for n in range(0, 6):
        cases.extend(itertools.product(range(8), repeat=n))
    rng = np.random.default_rng(1234 + b)
    cases.extend(tuple(r) for r in rng.integers(0, 8, size=(2000, 6)))
    for c in cases:
        keys = np.array(c, np.uint32)
        n = keys.size
        vals = np.arange(n, dtype=np.uint32)
        kout, vout = oracle.sort(keys, vals, 0, 3, b)
        pos = rank_positions(keys)
        ek = np.empty_like(keys)
        ev = np.empty_like(vals)
        ek[pos], ev[pos] = keys, vals
        assert kout.tolist() == ek.tolist(), (c, b)
        assert vout.tolist() == ev.tolist(), (c, b)


def test_brute_force_bit_ranges_u64():
    """Short u64 inputs sorted on a window of bits in the middle of the key:
    the bits outside the window ride along and do not order."""
    rng = np.random.default_rng(7)
    for trial in range(300):
        n = int(rng.integers(0, 40))
        keys = rng.integers(0, 2**63, size=n, dtype=np.uint64) * np.uint64(2) + \
            rng.integers(0, 2, size=n, dtype=np.uint64)
        begin = int(rng.integers(0, 60))
        end = int(rng.integers(begin + 1, 65))
        b = int(rng.integers(1, 9))
        kout, vout = oracle.sort(keys, np.arange(n, dtype=np.uint32), begin, end, b)
        pos = rank_positions(field(keys, begin, end).astype(object)) if end - begin == 64 \
            else rank_positions(field(keys, begin, end).astype(np.int64))
        ek = np.empty_like(keys)
        ek[pos] = keys
        assert kout.tolist() == ek.tolist(), (begin, end, b)


# -------------------------------------------------------------- library special

@pytest.mark.parametrize("dtype", [np.uint32, np.uint64])
@pytest.mark.parametrize("begin,end,b", [(0, None, 8), (0, None, 4), (0, None, 5),
                                         (3, 29, 7), (0, 12, 4), (8, 24, 3),
                                         (0, None, 1), (0, None, 11)])
def test_against_numpy_stable_argsort(dtype, begin, end, b):
    kb = 32 if dtype == np.uint32 else 64
    end = kb if end is None else end
    if kb == 64 and b == 1:
        pytest.skip("64 one-bit passes: covered by the brute-force test")
    n = 20011
    keys = workloads.words(3, 0, n)
    keys = (keys >> np.uint64(32)).astype(np.uint32) if dtype == np.uint32 else keys
    keys[::7] = keys[0]  # plenty of ties
    vals = workloads.index_payload(n)
    kout, vout = oracle.sort(keys, vals, begin, end, b)
    order = np.argsort(field(keys, begin, end), kind="stable")
    assert np.array_equal(kout, keys[order])
    assert np.array_equal(vout, vals[order])


@pytest.mark.parametrize("name", list(workloads.U32_DISTRIBUTIONS))
def test_invariants_u32_distributions(name):
    n = 50000
    keys = workloads.U32_DISTRIBUTIONS[name](n, 0)
    vals = workloads.index_payload(n)
    kout, vout = oracle.sort(keys, vals, 0, 32, 8)
    # permutation: payloads are a permutation of 0..n-1 and keys follow them
    assert np.array_equal(np.sort(vout), vals)
    assert np.array_equal(kout, keys[vout])
    # non-decreasing
    assert np.all(kout[1:] >= kout[:-1])
    # ties keep input order (payload = original index)
    tie = kout[1:] == kout[:-1]
    assert np.all(vout[1:][tie] > vout[:-1][tie])


def test_keys_only_and_empty():
    k, v = oracle.sort(np.array([], np.uint32))
    assert k.size == 0 and v is None
    k, v = oracle.sort(np.array([5, 1, 5, 0], np.uint32), None, 0, 32, 8)
    assert k.tolist() == [0, 1, 5, 5]


def test_invalid_ranges_rejected():
    keys = np.arange(4, dtype=np.uint32)
    for begin, end, b in [(0, 33, 8), (5, 5, 8), (-1, 8, 8), (0, 32, 0), (0, 32, 17)]:
        with pytest.raises(ValueError):
            oracle.sort(keys, None, begin, end, b)


# ------------------------------------------------------------------ histograms

@pytest.mark.parametrize("dtype,begin,end,b", [(np.uint32, 0, 32, 8), (np.uint32, 0, 32, 4),
                                               (np.uint64, 0, 64, 8), (np.uint64, 0, 40, 8),
                                               (np.uint32, 5, 30, 6)])
def test_pass_histograms_against_bincount(dtype, begin, end, b):
    n = 30000
    keys = workloads.words(5, 0, n)
    if dtype == np.uint32:
        keys = (keys >> np.uint64(32)).astype(np.uint32)
    hist = oracle.pass_histograms(keys, begin, end, b)
    P = -(-(end - begin) // b)
    assert hist.shape == (P, 1 << b)
    for p in range(P):
        shift = begin + p * b
        w = min(b, end - shift)
        d = field(keys, shift, shift + w).astype(np.int64)
        assert np.array_equal(hist[p], np.bincount(d, minlength=1 << b))
        assert int(hist[p].sum()) == n


# ------------------------------------------------------------ 16-bit float keys

def _f16_values():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)


def _bf16_values():
    return (np.arange(65536, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("decode", [_f16_values, _bf16_values], ids=["f16", "bf16"])
def test_order_key16_is_order_preserving_bijection(decode):
    t = np.array([oracle.order_key16(u) for u in range(65536)], np.int64)
    assert np.unique(t).size == 65536                       # bijection
    vals = decode()
    bits = np.arange(65536)
    finite_or_inf = ~np.isnan(vals)
    order = np.argsort(t)
    v = vals[order]
    b = bits[order]
    fin = finite_or_inf[order]
    # monotone on every non-NaN pattern
    vv = v[fin]
    assert np.all(vv[1:] >= vv[:-1])
    # equal values only for the two zeros: -0 sorts strictly before +0
    assert t[0x8000] < t[0x0000]
    assert t[0x8000] + 1 == t[0x0000]
    # NaNs: negative-sign ones before -inf, positive-sign ones after +inf
    nan_pos = np.nonzero(~fin)[0]
    neg_nan = nan_pos[(b[nan_pos] & 0x8000) != 0]
    pos_nan = nan_pos[(b[nan_pos] & 0x8000) == 0]
    first_finite = np.nonzero(fin)[0][0]
    last_finite = np.nonzero(fin)[0][-1]
    assert np.all(neg_nan < first_finite) and np.all(pos_nan > last_finite)
    assert np.isneginf(v[first_finite]) and np.isposinf(v[last_finite])


def test_order_key16_descending_is_complement():
    for u in range(0, 65536, 97):
        assert oracle.order_key16(u, True) == (~oracle.order_key16(u, False)) & 0xFFFF


@pytest.mark.parametrize("kind", ["f16", "bf16"])
@pytest.mark.parametrize("descending", [False, True])
def test_segmented_sort_against_numpy(kind, descending):
    x = workloads.rows16(6, 3001, kind=kind, seed=2)
    vals, idx = oracle.segmented_sort16(x, descending)
    t = np.array([oracle.order_key16(u, descending) for u in range(65536)], np.uint16)
    for r in range(x.shape[0]):
        order = np.argsort(t[x[r]], kind="stable")
        assert np.array_equal(idx[r], order)
        assert np.array_equal(vals[r], x[r][order])


def test_segmented_sort_float_order_without_nans():
    """On rows with no NaN the result is the float order, -0 before +0
    ascending (after it descending), ties in input order."""
    x = workloads.rows16(3, 2048, kind="f16", seed=9)
    x[x == workloads.F16_PNAN] = 0x3C00
    x[x == workloads.F16_NNAN] = 0xBC00
    f = x.view(np.float16).astype(np.float64)
    for desc in (False, True):
        vals, idx = oracle.segmented_sort16(x, desc)
        for r in range(3):
            v = vals[r].view(np.float16).astype(np.float64)
            assert np.all(v[1:] <= v[:-1]) if desc else np.all(v[1:] >= v[:-1])
            assert np.array_equal(vals[r], x[r][idx[r]])
            same = vals[r][1:] == vals[r][:-1]
            assert np.all(idx[r][1:][same] > idx[r][:-1][same])
            zeros = vals[r][(vals[r] == 0x0000) | (vals[r] == 0x8000)]
            first, second = (0x0000, 0x8000) if desc else (0x8000, 0x0000)
            k = int((zeros == first).sum())
            assert np.all(zeros[:k] == first) and np.all(zeros[k:] == second)
        assert np.array_equal(np.sort(f, axis=1), np.sort(vals.view(np.float16).astype(np.float64), axis=1))


def test_segmented_histograms_against_bincount():
    x = workloads.rows16(4, 5000, kind="bf16", seed=1)
    for desc in (False, True):
        h = oracle.segmented_histograms16(x, desc)
        t = np.array([oracle.order_key16(u, desc) for u in range(65536)], np.int64)
        for r in range(4):
            k = t[x[r]]
            assert np.array_equal(h[r, 0], np.bincount(k & 0xFF, minlength=256))
            assert np.array_equal(h[r, 1], np.bincount(k >> 8, minlength=256))
