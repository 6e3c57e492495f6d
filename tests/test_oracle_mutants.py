"""The pins catch plausible mistakes: each mutant is a copy of the oracle's C
source with one mistake planted (on the CPU), and at least one pin fails."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from tests.conftest import ROOT, read_golden
from lsd_radix_sort_gb300 import workloads

SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    # inclusive instead of exclusive scan (the "COMMON TRAP" of ch. 13.1)
    "inclusive_scan": ("    offsets[d] = sum;\n    sum += c;", "    sum += c;\n    offsets[d] = sum;"),
    # unstable walk: last element first into the ascending slots
    "reverse_walk": ("  for (size_t i = 0; i < n; i++) {\n    uint32_t d = digit[i];",
                     "  for (size_t i = n; i-- > 0;) {\n    uint32_t d = digit[i];"),
    # Listing 16-9 read literally: the window advances one bit per pass
    "shift_by_one": ("      int shift = begin_bit + p * b;                                           \\",
                     "      int shift = begin_bit + p;                                               \\"),
    # the narrower last digit dropped
    "floor_passes": ("return (end_bit - begin_bit + b - 1) / b;", "return (end_bit - begin_bit) / b;"),
    # MSD-first pass order
    "msd_order": ("      int shift = begin_bit + p * b;                                           \\\n      int w = pass_width(begin_bit, end_bit, b, p);                            \\\n      uint64_t mask = (w >= 64) ? ~0ull : ((1ull << w) - 1ull);                \\\n      const KEY_T",
                  "      int shift = begin_bit + (passes - 1 - p) * b;                            \\\n      int w = pass_width(begin_bit, end_bit, b, passes - 1 - p);               \\\n      uint64_t mask = (w >= 64) ? ~0ull : ((1ull << w) - 1ull);                \\\n      const KEY_T"),
    # sign handling of the float bijection forgotten for negatives
    "no_complement": ("(u & 0x8000u) ? (uint16_t)(~u)", "(u & 0x8000u) ? (uint16_t)(u)"),
    # descending flag ignored
    "no_descending": ("return descending ? (uint16_t)(~t) : t;", "return t;"),
    # exclusive scan off by one digit
    "scan_shift": ("for (uint32_t d = 0; d < radix; d++) counts[d] = 0;",
                   "for (uint32_t d = 0; d < radix; d++) counts[d] = (d == 1);"),
}


def build_mutant(tmp_path, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutant {name}: pattern not found"
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-o", str(so), str(c)],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    P, sz, i, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    lib.or_sort_u32.argtypes = [P, P, P, P, sz, i, i, i]
    lib.or_counting_pass.argtypes = [P, sz, u32, P, P, P]
    lib.or_order_key16.argtypes = [ctypes.c_uint16, i]
    lib.or_order_key16.restype = ctypes.c_uint16
    return lib


def pins_hold(lib):
    """A compact run of the pins; False as soon as one fails."""
    g = read_golden("base10_worked_example.txt")
    a = np.array(g["input"], np.uint32)
    digit = (a % 10).astype(np.uint32)
    counts = np.zeros(10, np.uint64)
    offs = np.zeros(10, np.uint64)
    dest = np.zeros(8, np.uint64)
    lib.or_counting_pass(digit.ctypes.data, 8, 10, counts.ctypes.data, offs.ctypes.data,
                         dest.ctypes.data)
    if offs.tolist() != g["place1_offsets"] or counts.tolist() != g["place1_counts"]:
        return False
    out = np.zeros(8, np.uint32)
    out[dest.astype(np.int64) % 8] = a
    if out.tolist() != g["pass1_values"]:
        return False
    # library special case with ties and a ragged last digit
    keys = (workloads.words(11, 0, 5000) >> np.uint64(44)).astype(np.uint32)  # 20 bits
    vals = np.arange(5000, dtype=np.uint32)
    ko, vo = np.zeros_like(keys), np.zeros_like(vals)
    lib.or_sort_u32(keys.ctypes.data, ko.ctypes.data, vals.ctypes.data, vo.ctypes.data,
                    5000, 0, 20, 8)
    order = np.argsort(keys, kind="stable")
    if not (np.array_equal(ko, keys[order]) and np.array_equal(vo, vals[order])):
        return False
    # float bijection order and its descending complement
    t = np.array([lib.or_order_key16(u, 0) for u in range(0, 65536, 3)], np.int64)
    f = (np.arange(0, 65536, 3, dtype=np.uint32).astype(np.uint16).view(np.float16)
         .astype(np.float64))
    ok = ~np.isnan(f)
    o = np.argsort(t[ok])
    if not np.all(np.diff(f[ok][o]) >= 0):
        return False
    if any(lib.or_order_key16(u, 1) != (~lib.or_order_key16(u, 0)) & 0xFFFF
           for u in range(0, 65536, 4099)):
        return False
    return True


def test_unmutated_oracle_passes(tmp_path):
    src = open(SRC).read()
    c = tmp_path / "clean.c"
    c.write_text(src)
    so = tmp_path / "clean.so"
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-o", str(so), str(c)],
                   check=True)
    lib = ctypes.CDLL(str(so))
    P, sz, i, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    lib.or_sort_u32.argtypes = [P, P, P, P, sz, i, i, i]
    lib.or_counting_pass.argtypes = [P, sz, u32, P, P, P]
    lib.or_order_key16.argtypes = [ctypes.c_uint16, i]
    lib.or_order_key16.restype = ctypes.c_uint16
    assert pins_hold(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    assert not pins_hold(build_mutant(tmp_path, name)), f"mutant {name} slipped through"
