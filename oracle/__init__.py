"""ORACLE -- test infrastructure, not product code.

Python access to the plain-C oracle in ``oracle.c`` (a single-threaded CPU
statement of LSD radix sort built from the three loops of a counting-sort
pass, CUDA Handbook ch. 16 "Radix Sort", Listings 16-8 and 16-9).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library; the two meet
only in the seeded input generators (``lsd_radix_sort_gb300.workloads``),
which hold none of the method's arithmetic.

``build()`` compiles ``oracle.c`` with the host C compiler into
``oracle/_build/liboracle.so``; the library is (re)built on first use when it
is missing or older than the source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

OR_OK = 0
OR_ERR_INVALID = 1
OR_ERR_NOMEM = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C99, -O2, no target-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        sz = ctypes.c_size_t
        i = ctypes.c_int
        i64 = ctypes.c_int64
        u32 = ctypes.c_uint32
        lib.or_histogram.argtypes = [P, sz, u32, P]
        lib.or_histogram.restype = None
        lib.or_exclusive_scan.argtypes = [P, u32, P]
        lib.or_exclusive_scan.restype = None
        lib.or_stable_destinations.argtypes = [P, sz, u32, P, P]
        lib.or_stable_destinations.restype = i
        lib.or_counting_pass.argtypes = [P, sz, u32, P, P, P]
        lib.or_counting_pass.restype = i
        lib.or_num_passes.argtypes = [i, i, i]
        lib.or_num_passes.restype = i
        for name in ("or_sort_u32", "or_sort_u64"):
            f = getattr(lib, name)
            f.argtypes = [P, P, P, P, sz, i, i, i]
            f.restype = i
        for name in ("or_pass_histograms_u32", "or_pass_histograms_u64"):
            f = getattr(lib, name)
            f.argtypes = [P, sz, i, i, i, P]
            f.restype = i
        lib.or_order_key16.argtypes = [ctypes.c_uint16, i]
        lib.or_order_key32.argtypes = [ctypes.c_uint32, i, i]
        lib.or_order_key32.restype = ctypes.c_uint32
        lib.or_order_key64.argtypes = [ctypes.c_uint64, i, i]
        lib.or_order_key64.restype = ctypes.c_uint64
        for name in ("or_sort_typed32", "or_sort_typed64"):
            f = getattr(lib, name)
            f.argtypes = [P, P, P, P, sz, i, i, i, i, i]
        lib.or_order_key16.restype = ctypes.c_uint16
        lib.or_segmented_sort16.argtypes = [P, P, P, i64, i64, i]
        lib.or_segmented_sort16.restype = i
        lib.or_segmented_histograms16.argtypes = [P, i64, i64, i, P]
        lib.or_segmented_histograms16.restype = i
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _check(rc: int, what: str):
    if rc != OR_OK:
        raise ValueError(f"oracle {what} failed with code {rc}")


def counting_pass(digit: np.ndarray, radix: int):
    """One stable counting-sort pass over precomputed digits.

    Returns (counts, offsets, dest): the digit histogram, its exclusive scan
    and the destination of every element (Listing 16-8's three loops).
    """
    lib = _load()
    digit = np.ascontiguousarray(digit, dtype=np.uint32)
    n = digit.size
    counts = np.zeros(radix, np.uint64)
    offsets = np.zeros(radix, np.uint64)
    dest = np.zeros(max(n, 1), np.uint64)[:n]
    _check(lib.or_counting_pass(_ptr(digit), n, radix, _ptr(counts),
                                _ptr(offsets), _ptr(dest) if n else None),
           "counting_pass")
    return counts, offsets, dest


def num_passes(begin_bit: int, end_bit: int, digit_bits: int) -> int:
    return int(_load().or_num_passes(begin_bit, end_bit, digit_bits))


def sort(keys: np.ndarray, values: np.ndarray | None = None, begin_bit: int = 0,
         end_bit: int | None = None, digit_bits: int = 8):
    """Stable LSD sort of u32 or u64 keys on bits [begin_bit, end_bit).

    ``values`` (u32 or None) ride along.  Returns (keys_out, values_out).
    """
    lib = _load()
    keys = np.ascontiguousarray(keys)
    if keys.dtype == np.uint32:
        f, kb = lib.or_sort_u32, 32
    elif keys.dtype == np.uint64:
        f, kb = lib.or_sort_u64, 64
    else:
        raise TypeError(f"oracle sort: unsupported key dtype {keys.dtype}")
    if end_bit is None:
        end_bit = kb
    n = keys.size
    kout = np.empty_like(keys)
    vout = None
    if values is not None:
        values = np.ascontiguousarray(values, dtype=np.uint32)
        if values.size != n:
            raise ValueError("values must have one entry per key")
        vout = np.empty_like(values)
    _check(f(_ptr(keys), _ptr(kout), _ptr(values), _ptr(vout), n, begin_bit,
             end_bit, digit_bits), "sort")
    return kout, vout


def pass_histograms(keys: np.ndarray, begin_bit: int = 0, end_bit: int | None = None,
                    digit_bits: int = 8) -> np.ndarray:
    """Digit histogram of every pass, shape (passes, 2**digit_bits), u64."""
    lib = _load()
    keys = np.ascontiguousarray(keys)
    if keys.dtype == np.uint32:
        f, kb = lib.or_pass_histograms_u32, 32
    elif keys.dtype == np.uint64:
        f, kb = lib.or_pass_histograms_u64, 64
    else:
        raise TypeError(f"oracle histograms: unsupported key dtype {keys.dtype}")
    if end_bit is None:
        end_bit = kb
    p = num_passes(begin_bit, end_bit, digit_bits)
    hist = np.zeros((max(p, 1), 1 << digit_bits), np.uint64)
    _check(f(_ptr(keys), keys.size, begin_bit, end_bit, digit_bits, _ptr(hist)),
           "pass_histograms")
    return hist[:p]


_TYPES = {"u32": (0, 4), "i32": (1, 4), "f32": (2, 4), "u64": (0, 8), "i64": (1, 8),
          "f64": (2, 8)}


def order_key(bits: int, key_type: str, descending: bool = False) -> int:
    """T(k) of one 32/64-bit pattern under the typed bijection."""
    code, size = _TYPES[key_type]
    lib = _load()
    f = lib.or_order_key32 if size == 4 else lib.or_order_key64
    return int(f(bits & ((1 << (8 * size)) - 1), code, int(bool(descending))))


def sort_typed(keys: np.ndarray, key_type: str, values: np.ndarray | None = None,
               descending: bool = False, begin_bit: int = 0, end_bit: int | None = None,
               digit_bits: int = 8):
    """Stable sort of typed keys (any 4- or 8-byte dtype, read as bit
    patterns) by the bits [begin_bit, end_bit) of T(k).  Returns
    (keys_out in the input dtype, values_out)."""
    code, size = _TYPES[key_type]
    keys = np.ascontiguousarray(keys)
    if keys.dtype.itemsize != size:
        raise TypeError(f"{key_type} keys are {size}-byte, got {keys.dtype}")
    bits_t = np.uint32 if size == 4 else np.uint64
    kin = keys.view(bits_t)
    lib = _load()
    f = lib.or_sort_typed32 if size == 4 else lib.or_sort_typed64
    end_bit = 8 * size if end_bit is None else end_bit
    kout = np.empty_like(kin)
    vout = None
    if values is not None:
        values = np.ascontiguousarray(values, dtype=np.uint32)
        if values.size != kin.size:
            raise ValueError("values must have one entry per key")
        vout = np.empty_like(values)
    _check(f(_ptr(kin), _ptr(kout), _ptr(values), _ptr(vout), kin.size, code,
             int(bool(descending)), begin_bit, end_bit, digit_bits), "sort_typed")
    return kout.view(keys.dtype), vout


def order_key16(bits: int, descending: bool = False) -> int:
    return int(_load().or_order_key16(bits & 0xFFFF, int(bool(descending))))


def segmented_sort16(x: np.ndarray, descending: bool = False):
    """Row-wise stable sort of a (rows, cols) array of 16-bit float patterns.

    Returns (sorted bit patterns as uint16, int64 column indices).
    """
    lib = _load()
    x = np.ascontiguousarray(x).view(np.uint16)
    if x.ndim != 2:
        raise ValueError("segmented_sort16 expects a 2-D array")
    rows, cols = x.shape
    vals = np.empty_like(x)
    idx = np.empty((rows, cols), np.int64)
    _check(lib.or_segmented_sort16(_ptr(x), _ptr(vals), _ptr(idx), rows, cols,
                                   int(bool(descending))), "segmented_sort16")
    return vals, idx


def segmented_histograms16(x: np.ndarray, descending: bool = False) -> np.ndarray:
    """Per-row digit histograms of both passes, shape (rows, 2, 256), u64."""
    lib = _load()
    x = np.ascontiguousarray(x).view(np.uint16)
    rows, cols = x.shape
    hist = np.zeros((rows, 2, 256), np.uint64)
    _check(lib.or_segmented_histograms16(_ptr(x), rows, cols, int(bool(descending)),
                                         _ptr(hist)), "segmented_histograms16")
    return hist
