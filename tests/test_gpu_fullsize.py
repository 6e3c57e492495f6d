"""Full-size parity (2^28 keys) in the launch configuration bench.py times.

The oracle's full run would take minutes per case here, so the result is
checked through properties that together fix the unique stable sort, plus
sampled positions computed one by one from the closed form
    pos(i) = #{j : f(k_j) < f(k_i)} + #{j < i : f(k_j) = f(k_i)}:
  * the sort field is non-decreasing;
  * the payloads (original indices) form a permutation and every output key
    is the input key its payload points at;
  * equal sort fields keep increasing payloads (stability).
"""
import numpy as np
import pytest
import torch

from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import field, to_dev, to_host

pytestmark = pytest.mark.gpu

N = 1 << 28


def check_sorted_pairs(keys, vals_out, keys_out, begin, end, samples=6, seed=0):
    n = keys.size
    f_out = field(keys_out, begin, end) if end - begin < keys.dtype.itemsize * 8 else keys_out
    assert np.all(f_out[1:] >= f_out[:-1]), "sort field decreases"
    seen = np.zeros(n, dtype=bool)
    seen[vals_out] = True
    assert seen.all(), "payloads are not a permutation"
    assert np.array_equal(keys[vals_out], keys_out), "keys do not follow their payloads"
    tie = f_out[1:] == f_out[:-1]
    assert np.all(vals_out[1:][tie] > vals_out[:-1][tie]), "ties out of input order"
    f_in = field(keys, begin, end) if end - begin < keys.dtype.itemsize * 8 else keys
    rng = np.random.default_rng(seed)
    for i in rng.integers(0, n, samples):
        k = f_in[i]
        pos = int(np.count_nonzero(f_in < k)) + int(np.count_nonzero(f_in[:i] == k))
        assert vals_out[pos] == i and keys_out[pos] == keys[i], f"sampled rank of input {i}"


@pytest.mark.parametrize("dist", list(workloads.U32_DISTRIBUTIONS))
def test_u32_pairs_2p28(rs, dist):
    keys = workloads.U32_DISTRIBUTIONS[dist](N, 0)
    vals = workloads.index_payload(N)
    dk, dv = to_dev(keys), to_dev(vals)
    temp = torch.empty(rs.temp_bytes(N, 4, 4, 0, 32, 8), dtype=torch.uint8, device="cuda")
    ko, vo = rs.radix_sort_pairs(dk, dv, begin_bit=0, end_bit=32, digit_bits=8, temp=temp)
    assert rs.device_status(temp) == rs.RS_OK
    del dk, dv
    check_sorted_pairs(keys, to_host(vo, np.uint32), to_host(ko, np.uint32), 0, 32)


@pytest.mark.parametrize("dist,begin,end", [("uniform", 0, 64), ("skewed", 0, 64),
                                            ("uniform", 0, 40)])
def test_u64_pairs_2p28(rs, dist, begin, end):
    keys = workloads.U64_DISTRIBUTIONS[dist](N, 0)
    vals = workloads.index_payload(N)
    dk, dv = to_dev(keys), to_dev(vals)
    temp = torch.empty(rs.temp_bytes(N, 8, 4, begin, end, 8), dtype=torch.uint8, device="cuda")
    ko, vo = rs.radix_sort_pairs(dk, dv, begin_bit=begin, end_bit=end, digit_bits=8, temp=temp)
    assert rs.device_status(temp) == rs.RS_OK
    del dk, dv
    check_sorted_pairs(keys, to_host(vo, np.uint32), to_host(ko, np.uint64), begin, end)


def test_u32_pairs_above_2p30(rs):
    """2^30 + 12,345 keys: past the 30-bit count of a 32-bit look-back word, so
    the look-back runs on 64-bit words.  Checked on the device by the same
    properties, plus sampled closed-form ranks."""
    n = (1 << 30) + 12345
    keys = workloads.u32_uniform(n, 1)
    dk = to_dev(keys)
    dv = to_dev(workloads.index_payload(n))
    del keys
    temp = torch.empty(rs.temp_bytes(n, 4, 4, 0, 32, 8), dtype=torch.uint8, device="cuda")
    ko, vo = rs.radix_sort_pairs(dk, dv, temp=temp)
    assert rs.device_status(temp) == rs.RS_OK
    del temp, dv
    flip = torch.tensor(-(1 << 31), dtype=torch.int32, device="cuda")
    ks = ko ^ flip  # unsigned order as signed order
    assert bool((ks[1:] >= ks[:-1]).all()), "keys decrease"
    ties = ks[1:] == ks[:-1]
    assert bool((vo[1:][ties] > vo[:-1][ties]).all()), "ties out of input order"
    del ks, ties
    idx = vo.long()  # payloads are input positions below 2^31
    assert torch.equal(dk[idx], ko), "keys do not follow their payloads"
    seen = torch.zeros(n, dtype=torch.bool, device="cuda")
    seen[idx] = True
    assert bool(seen.all()), "payloads are not a permutation"
    del seen, idx
    dks = dk ^ flip
    rng = np.random.default_rng(3)
    for i in [0, n - 1, *rng.integers(0, n, 4).tolist()]:
        k = dks[i]
        pos = int((dks < k).sum()) + int((dks[:i] == k).sum())
        assert int(vo[pos]) == i and int(ko[pos]) == int(dk[i]), f"sampled rank of input {i}"


def _const_byte_keys(n, seed):
    # bits 8..15 constant: with pass skipping three of four passes run
    return (workloads.u32_uniform(n, seed) & np.uint32(0xFFFF00FF)) | np.uint32(0x5A00)


@pytest.mark.parametrize("case", ["keys_only", "pairs_pass_skipping"])
def test_u32_above_2p30_keys_and_skipping(rs, case):
    """The 64-bit look-back words with keys only (checked against the sorted
    multiset), and with pass skipping (the device-side schedule) checked by
    the properties above."""
    n = (1 << 30) + 777
    flip = torch.tensor(-(1 << 31), dtype=torch.int32, device="cuda")
    if case == "keys_only":
        dk = to_dev(workloads.u32_uniform(n, 2))
        temp = torch.empty(rs.temp_bytes(n, 4, 0, 0, 32, 8), dtype=torch.uint8, device="cuda")
        ko = rs.radix_sort_keys(dk, temp=temp)
        assert rs.device_status(temp) == rs.RS_OK
        del temp
        want = torch.sort(dk ^ flip).values
        assert torch.equal(ko ^ flip, want)
        return
    dk = to_dev(_const_byte_keys(n, 3))
    dv = to_dev(workloads.index_payload(n))
    temp = torch.empty(rs.temp_bytes(n, 4, 4, 0, 32, 8), dtype=torch.uint8, device="cuda")
    ko, vo = rs.radix_sort_pairs(dk, dv, temp=temp, pass_skipping=True)
    assert rs.device_status(temp) == rs.RS_OK and rs.passes_run(temp) == 3
    del temp, dv
    ks = ko ^ flip
    assert bool((ks[1:] >= ks[:-1]).all()), "keys decrease"
    ties = ks[1:] == ks[:-1]
    assert bool((vo[1:][ties] > vo[:-1][ties]).all()), "ties out of input order"
    del ks, ties
    idx = vo.long()
    assert torch.equal(dk[idx], ko), "keys do not follow their payloads"
    seen = torch.zeros(n, dtype=torch.bool, device="cuda")
    seen[idx] = True
    assert bool(seen.all()), "payloads are not a permutation"
