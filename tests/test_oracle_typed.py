"""Pins of the oracle's typed sorts (signed and floating-point keys, both
directions) against numpy's stable argsort and against the special-value
order that the bijection defines ("100 Days of GPU", day 35, Pitfalls: a
radix sort orders bit patterns, so signed and float keys go through a
bijection on the way in).  Each planted mistake in the typed code fails at
least one pin."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests.conftest import ROOT
from lsd_radix_sort_gb300 import workloads

SRC = os.path.join(ROOT, "oracle", "oracle.c")


def _stable(x):
    return np.argsort(x, kind="stable")


def _keys_i32(n, seed):
    w = workloads.words(seed, 0, n)
    k = (w >> np.uint64(32)).astype(np.uint32).view(np.int32)
    k[::5] = k[0]  # ties
    return k


def _keys_f(n, seed, dtype):
    w = workloads.words(seed, 1, n)
    x = ((w >> np.uint64(11)).astype(np.float64) / 2.0**53 - 0.5) * 1e6
    x = x.astype(dtype)
    x[::7] = x[1]          # ties
    x[x == 0] = 0          # no -0.0 (numpy orders it equal to +0.0)
    return x


def _check(keys, key_type, descending, expect_order):
    vals = np.arange(keys.size, dtype=np.uint32)
    ko, vo = oracle.sort_typed(keys, key_type, vals, descending)
    assert np.array_equal(vo, expect_order.astype(np.uint32))
    assert np.array_equal(ko.view(np.uint8), keys[expect_order].view(np.uint8))


@pytest.mark.parametrize("descending", [False, True])
def test_i32_matches_numpy(descending):
    k = _keys_i32(20_000, 5)
    k[3] = np.iinfo(np.int32).min
    k[4] = np.iinfo(np.int32).max
    # ~x reverses the order of two's-complement integers without overflow
    order = _stable(~k) if descending else _stable(k)
    _check(k, "i32", descending, order)


@pytest.mark.parametrize("descending", [False, True])
def test_i64_matches_numpy(descending):
    w = workloads.words(6, 0, 20_000)
    k = w.view(np.int64).copy()
    k[::4] = k[2]
    k[5] = np.iinfo(np.int64).min
    order = _stable(~k) if descending else _stable(k)
    _check(k, "i64", descending, order)


@pytest.mark.parametrize("dtype,key_type", [(np.float32, "f32"), (np.float64, "f64")])
@pytest.mark.parametrize("descending", [False, True])
def test_float_matches_numpy(dtype, key_type, descending):
    x = _keys_f(20_000, 7, dtype)
    x[10], x[11] = np.inf, -np.inf
    order = _stable(-x) if descending else _stable(x)
    _check(x, key_type, descending, order)


@pytest.mark.parametrize("descending", [False, True])
def test_unsigned_typed_is_plain_sort(descending):
    k = workloads.u32_uniform(10_000, 8)
    k[::3] = k[1]
    order = _stable(~k) if descending else _stable(k)
    _check(k, "u32", descending, order)
    k64 = workloads.u64_uniform(10_000, 9)
    order = _stable(~k64) if descending else _stable(k64)
    _check(k64, "u64", descending, order)


# Special values, ascending, by the rule: negative patterns complemented,
# others with the sign bit set.  So a NaN with the sign bit set precedes
# -inf, -0.0 precedes +0.0, and a NaN with the sign bit clear follows +inf.
F32_ASCENDING = [0xFFC00000,  # -NaN
                 0xFF800000,  # -inf
                 0xFF7FFFFF,  # -max
                 0xBF800000,  # -1
                 0x80000001,  # -smallest subnormal
                 0x80000000,  # -0
                 0x00000000,  # +0
                 0x00000001,  # +smallest subnormal
                 0x3F800000,  # 1
                 0x7F7FFFFF,  # max
                 0x7F800000,  # +inf
                 0x7FC00000]  # +NaN
F64_ASCENDING = [0xFFF8000000000000, 0xFFF0000000000000, 0xFFEFFFFFFFFFFFFF,
                 0xBFF0000000000000, 0x8000000000000001, 0x8000000000000000,
                 0x0000000000000000, 0x0000000000000001, 0x3FF0000000000000,
                 0x7FEFFFFFFFFFFFFF, 0x7FF0000000000000, 0x7FF8000000000000]


@pytest.mark.parametrize("pats,bits_t,key_type", [(F32_ASCENDING, np.uint32, "f32"),
                                                  (F64_ASCENDING, np.uint64, "f64")])
@pytest.mark.parametrize("descending", [False, True])
def test_float_special_values(pats, bits_t, key_type, descending):
    want = np.array(pats, dtype=bits_t)
    if descending:
        want = want[::-1]
    shuffled = np.array(pats, dtype=bits_t)[[5, 0, 11, 3, 8, 1, 10, 6, 2, 9, 4, 7]]
    ko, _ = oracle.sort_typed(shuffled, key_type, None, descending)
    assert np.array_equal(ko, want)


def test_ties_keep_input_order_both_directions():
    k = np.array([2, -1, 2, -1, 0, 2], dtype=np.int32)
    vals = np.arange(6, dtype=np.uint32)
    _, va = oracle.sort_typed(k, "i32", vals, False)
    _, vd = oracle.sort_typed(k, "i32", vals, True)
    assert va.tolist() == [1, 3, 4, 0, 2, 5]
    assert vd.tolist() == [0, 2, 5, 4, 1, 3]


def test_bit_range_of_the_transformed_key():
    k = _keys_i32(10_000, 10)
    t = k.view(np.uint32) ^ np.uint32(0x80000000)  # signed -> unsigned order
    field = (t >> np.uint32(8)) & np.uint32(0xFFFF)
    vals = np.arange(k.size, dtype=np.uint32)
    _, vo = oracle.sort_typed(k, "i32", vals, False, 8, 24, 5)
    assert np.array_equal(vo, _stable(field).astype(np.uint32))


# ------------------------------------------------------------ mutants

MUTANTS = {
    "signed_no_flip": ("if (type == OR_SIGNED) t = k ^ sign;\n  if (type == OR_FLOAT) t = (k & sign) ? ~k : (k | sign);\n  return descending ? ~t : t;\n}\n\nuint64_t",
                       "if (type == OR_SIGNED) t = k;\n  if (type == OR_FLOAT) t = (k & sign) ? ~k : (k | sign);\n  return descending ? ~t : t;\n}\n\nuint64_t"),
    "float_no_complement": ("if (type == OR_FLOAT) t = (k & sign) ? ~k : (k | sign);\n  return descending ? ~t : t;\n}\n\nuint64_t",
                            "if (type == OR_FLOAT) t = (k & sign) ? k : (k | sign);\n  return descending ? ~t : t;\n}\n\nuint64_t"),
    "desc_ignored": ("  return descending ? ~t : t;\n}\n\nuint64_t", "  return t;\n}\n\nuint64_t"),
    "no_gather": ("keys_out[i] = keys_in[order[i]];", "keys_out[i] = keys_in[i];"),
}


def _mutant(tmp_path, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutant {name}: pattern not found once"
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-o", str(so), str(c)],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    P, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.or_sort_typed32.argtypes = [P, P, P, P, sz, i, i, i, i, i]
    return lib


def _pins_hold(lib):
    def run(keys, code, desc):
        kin = np.ascontiguousarray(keys).view(np.uint32)
        kout = np.empty_like(kin)
        vals = np.arange(kin.size, dtype=np.uint32)
        vout = np.empty_like(vals)
        rc = lib.or_sort_typed32(kin.ctypes.data, kout.ctypes.data, vals.ctypes.data,
                                 vout.ctypes.data, kin.size, code, desc, 0, 32, 8)
        return rc, kout, vout
    k = _keys_i32(3000, 11)
    for desc in (0, 1):
        rc, ko, vo = run(k, 1, desc)
        order = _stable(~k) if desc else _stable(k)
        if rc != 0 or not np.array_equal(vo, order) or not np.array_equal(ko.view(np.int32), k[order]):
            return False
    x = _keys_f(3000, 12, np.float32)
    for desc in (0, 1):
        rc, ko, vo = run(x, 2, desc)
        order = _stable(-x) if desc else _stable(x)
        if rc != 0 or not np.array_equal(vo, order):
            return False
    return True


def test_pins_hold_for_the_oracle(tmp_path):
    assert _pins_hold(_mutant_identity(tmp_path))


def _mutant_identity(tmp_path):
    c = tmp_path / "same.c"
    so = tmp_path / "same.so"
    c.write_text(open(SRC).read())
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-o", str(so), str(c)],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    P, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.or_sort_typed32.argtypes = [P, P, P, P, sz, i, i, i, i, i]
    return lib


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    assert not _pins_hold(_mutant(tmp_path, name))
