"""The parity helper's diagnostics, on host arrays (no GPU): it accepts the
oracle's own result and names the fault in broken ones."""
import numpy as np
import pytest

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import assert_pairs


def _case():
    keys = workloads.u32_small(3000, 9, 6)  # many ties
    vals = workloads.index_payload(keys.size)
    return oracle.sort(keys, vals, 0, 32, 8)


def test_accepts_the_oracle():
    ek, ev = _case()
    assert_pairs(ek, ev, ek, ev)
    assert_pairs(ek, None, ek, None)


def test_names_a_key_fault():
    ek, ev = _case()
    k = ek.copy()
    k[[10, 2000]] = k[[2000, 10]]
    with pytest.raises(AssertionError, match="keys differ at 10 "):
        assert_pairs(k, ev, ek, ev)


def test_names_a_stability_fault():
    ek, ev = _case()
    i = int(np.flatnonzero(ek[1:] == ek[:-1])[0])
    v = ev.copy()
    v[[i, i + 1]] = v[[i + 1, i]]
    with pytest.raises(AssertionError, match="stability"):
        assert_pairs(ek, v, ek, ev)


def test_names_a_payload_that_left_its_key():
    ek, ev = _case()
    j = int(np.flatnonzero(ek != ek[0])[0])
    v = ev.copy()
    v[[0, j]] = v[[j, 0]]
    with pytest.raises(AssertionError, match="did not travel"):
        assert_pairs(ek, v, ek, ev)
