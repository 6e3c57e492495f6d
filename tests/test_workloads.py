"""The seeded input generators: SplitMix64 in counter mode and the recipes."""
import numpy as np

from lsd_radix_sort_gb300 import workloads


def test_splitmix64_published_sequence():
    # SplitMix64 started from state 0 (Vigna's splitmix64.c) begins with these.
    assert workloads.word(0, 0, 0) == 0xE220A8397B1DCDAF
    assert workloads.word(0, 0, 1) == 0x6E789E6AA1B965F4
    w = workloads.words(0, 0, 2)
    assert [int(x) for x in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_chunked_generation_matches_scalar():
    n = (1 << 22) + 12345   # crosses the chunk size
    w = workloads.words(7, 3, n)
    for i in (0, 1, (1 << 22) - 1, 1 << 22, n - 1):
        assert int(w[i]) == workloads.word(7, 3, i)
    w2 = workloads.words(7, 3, 10, start=(1 << 22) - 5)
    assert np.array_equal(w2, w[(1 << 22) - 5:(1 << 22) + 5])


def test_recipes():
    n = 1 << 16
    small = workloads.u32_small(1024, 0, 12)
    assert small.max() < 4096 and small.dtype == np.uint32
    assert np.all(workloads.u32_all_equal(n) == workloads.word(0, 0, 0) >> 32)
    le = workloads.u32_low_entropy(n)
    ones = np.unpackbits(le.view(np.uint8)).mean()
    assert 0.04 < ones < 0.09          # each bit set with probability 1/16
    s = workloads.u32_sorted(n)
    assert np.all(s[1:] >= s[:-1])
    r = workloads.u32_reverse_sorted(n)
    assert np.array_equal(r, s[::-1])
    sk = workloads.u64_skewed(n)
    assert sk.dtype == np.uint64 and np.median(sk.astype(np.float64)) < 2.0 ** 64 * 0.5 ** 8 * 1.1


def test_rows16_mix():
    x = workloads.rows16(8, 4096, "f16", seed=0)
    f = x.view(np.float16).astype(np.float64)
    n = x.size
    for pat in (0x0000, 0x8000, 0x7C00, 0xFC00):
        frac = (x == pat).sum() / n
        assert 0.006 < frac < 0.014, hex(pat)
    nanfrac = np.isnan(f).mean()
    assert 0.006 < nanfrac < 0.014
    fin = f[np.isfinite(f)]
    assert abs(fin.mean()) < 0.05 and 0.9 < fin.std() < 1.1
    b = workloads.rows16(2, 1000, "bf16", seed=0)
    assert ((b == 0x7F80).sum() + (b == 0xFF80).sum()) > 0


def test_bf16_rounding_nearest_even():
    # exact bf16 values stay, halfway cases go to even
    x = np.array([1.0, 1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -2.5, 1.0 + 2.0**-8 + 2.0**-40])
    got = workloads.double_to_bf16_bits(x)
    assert got.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]
