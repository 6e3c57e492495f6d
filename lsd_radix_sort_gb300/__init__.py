"""GB300-native LSD radix sort: Python binding of the C-ABI library.

The sort itself runs entirely in ``liblsdrs.so`` (hand-written sm_103a CUDA
kernels behind the C ABI declared in ``include/lsdrs.h``).  This module only
marshals arguments: it takes PyTorch CUDA tensors, allocates outputs and the
scratch buffer with PyTorch, and passes raw device pointers and the current
stream to the library.  There is no fallback: if the library is missing or
fails to load, every call raises.

Keys may be given as 4-byte or 8-byte tensors; by default their bits are
sorted as unsigned integers, and ``key_type`` ("i32", "f32", "i64", "f64",
"u32", "u64") with ``descending`` selects the typed sorts.  Payloads are
4-byte tensors.  Modes (pass skipping, precomputed tile offsets, the
one-kernel path for short rows, the look-back wait limit) are keyword
arguments of each call: the library holds no
mode state, so calls on different threads or streams never affect each
other.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "RadixSortError", "load_library", "library_path", "temp_bytes", "radix_sort_keys",
    "radix_sort_pairs", "segmented_sort", "segmented_temp_bytes", "upfront_histograms",
    "device_status", "passes_run", "SMALL_SORT_MAX_KEYS", "copy_probe",
    "lookback_timeout_probe", "profile_enable", "profile_read", "launch_count_reset",
    "noalloc_status", "noalloc_timeout_probe", "EXPORTED_SYMBOLS", "RS_MAX_KEYS", "RS_MAX_ROW_KEYS", "checked_build",
    "BoundsViolation",
]

RS_OK, RS_ERR_INVALID, RS_ERR_TEMP_TOO_SMALL, RS_ERR_CUDA, RS_ERR_LOOKBACK_TIMEOUT = range(5)
RS_F16, RS_BF16 = 0, 1
KEY_TYPES = {"u32": (0, 4), "i32": (1, 4), "f32": (2, 4), "u64": (3, 8), "i64": (4, 8),
             "f64": (5, 8)}
RS_MAX_KEYS = (1 << 32) - 1       # one flat sort
RS_MAX_ROW_KEYS = (1 << 30) - 1   # one row of a row-wise sort
RS_OPT_PASS_SKIPPING, RS_OPT_TILE_OFFSETS, RS_OPT_NO_SMALL_SORT = 0x1, 0x2, 0x4
# Rows (or flat inputs) of at most this many keys, with 4- or 8-bit digits,
# are sorted by one kernel that runs every pass in shared memory (unless a
# call passes small_sort=False); it runs every pass, pass skipping included.
SMALL_SORT_MAX_KEYS = 8192
KERNEL_NAMES = {0: "upfront_hist", 1: "digit_scan", 2: "onesweep", 3: "copy_probe",
                4: "timeout_probe", 5: "finish", 6: "tile_counts",
                7: "small_sort"}

EXPORTED_SYMBOLS = (
    "radix_sort_keys_temp_bytes", "radix_sort_keys_u32", "radix_sort_keys_u64",
    "radix_sort_pairs_u32", "radix_sort_pairs_u64", "radix_segmented_sort_temp_bytes",
    "radix_segmented_sort_f16", "radix_segmented_sort_f16_ex", "radix_sort_histograms",
    "radix_sort_device_status", "rs_status_string", "rs_lookback_timeout_probe",
    "rs_copy_probe", "rs_profile_enable", "rs_profile_read", "rs_launch_count_reset",
    "radix_sort_pairs_u32_noalloc", "radix_sort_pairs_u32_noalloc_status",
    "rs_noalloc_timeout_probe", "radix_sort_keys_typed", "radix_sort_pairs_typed", "radix_sort_passes_run",
    "rs_checked_build", "radix_sort_checked_violations",
)


class RadixSortError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_status_name(status)}")


class KernelTime(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("ms", ctypes.c_float), ("units", ctypes.c_uint64)]


class Options(ctypes.Structure):
    """struct rs_options of include/lsdrs.h."""
    _fields_ = [("flags", ctypes.c_uint), ("lookback_timeout_ns", ctypes.c_uint64)]


def _options(pass_skipping=False, tile_offsets=False, small_sort=True, lookback_timeout_ns=0):
    """An rs_options for the call, or None when every option is at its default."""
    flags = ((RS_OPT_PASS_SKIPPING if pass_skipping else 0)
             | (RS_OPT_TILE_OFFSETS if tile_offsets else 0)
             | (0 if small_sort else RS_OPT_NO_SMALL_SORT))
    if not flags and not lookback_timeout_ns:
        return None
    return Options(flags, int(lookback_timeout_ns))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """The in-tree library, or the one named by LSDRS_LIB (tuning builds)."""
    return os.environ.get("LSDRS_LIB") or _build.LIB


def load_library() -> ctypes.CDLL:
    """Load liblsdrs.so (built by ``lsd_radix_sort_gb300.build``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m lsd_radix_sort_gb300.build` "
                "(there is no CPU fallback)")
        try:  # share the CUDA runtime PyTorch already loaded, when it is present
            import torch  # noqa: F401
        except Exception:
            pass
        lib = ctypes.CDLL(path)
        P, sz, i, i64, u64 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64,
                              ctypes.c_uint64)
        st = ctypes.c_int
        sig = {
            "radix_sort_keys_temp_bytes": [sz, i, i, i, i, i, P],
            "radix_sort_keys_u32": [P, P, sz, i, i, i, P, sz, P],
            "radix_sort_keys_u64": [P, P, sz, i, i, i, P, sz, P],
            "radix_sort_pairs_u32": [P, P, P, P, sz, i, i, i, P, sz, P],
            "radix_sort_pairs_u64": [P, P, P, P, sz, i, i, i, P, sz, P],
            "radix_segmented_sort_temp_bytes": [i64, i64, P],
            "radix_segmented_sort_f16": [P, P, P, i64, i64, i, i, P, sz, P],
            "radix_segmented_sort_f16_ex": [P, P, P, i64, i64, i, i, P, sz, P, P],
            "radix_sort_histograms": [P, i, sz, i, i, i, P, P, P, sz, P],
            "radix_sort_device_status": [P, P],
            "rs_lookback_timeout_probe": [P, u64, P, P],
            "rs_copy_probe": [P, P, sz, P],
            "rs_profile_enable": [i],
            "radix_sort_pairs_u32_noalloc": [P, P, P, P, sz, i, i, i, P],
            "radix_sort_pairs_u32_noalloc_status": [P],
            "rs_noalloc_timeout_probe": [u64, P, P],
            "radix_sort_keys_typed": [i, i, P, P, sz, i, i, i, P, sz, P, P],
            "radix_sort_passes_run": [P, P, P],
            "radix_sort_pairs_typed": [i, i, P, P, P, P, sz, i, i, i, P, sz, P, P],
            "radix_sort_checked_violations": [P, P, P, P],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = st
        lib.rs_status_string.argtypes = [st]
        lib.rs_status_string.restype = ctypes.c_char_p
        lib.rs_profile_read.argtypes = [P, i]
        lib.rs_profile_read.restype = i
        lib.rs_launch_count_reset.argtypes = []
        lib.rs_launch_count_reset.restype = u64
        lib.rs_checked_build.argtypes = []
        lib.rs_checked_build.restype = i
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    try:
        return load_library().rs_status_string(status).decode()
    except Exception:
        return f"status {status}"


def _check(status: int, what: str):
    if status != RS_OK:
        raise RadixSortError(status, what)


class BoundsViolation(RuntimeError):
    """A bounds-checked build recorded failed index tests during a sort."""


def checked_build() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(load_library().rs_checked_build())


def _violations(t, stream):
    count, site = ctypes.c_uint32(0), ctypes.c_uint32(0)
    _check(load_library().radix_sort_checked_violations(_ptr(t), _stream_ptr(stream),
                                                        ctypes.byref(count), ctypes.byref(site)),
           "radix_sort_checked_violations")
    return count.value, site.value


class _BoundsGuard:
    """Around one sort with a bounds-checked library: clear the scratch's
    violation words before, raise BoundsViolation if any test failed."""

    def __init__(self, t, stream, what):
        self.t, self.stream, self.what = t, stream, what
        self.on = checked_build()

    def __enter__(self):
        if self.on:
            _violations(self.t, self.stream)
        return self

    def __exit__(self, *exc):
        if self.on and exc[0] is None:
            count, site = _violations(self.t, self.stream)
            if count:
                raise BoundsViolation(f"{self.what}: {count} index tests failed "
                                      f"(first at site {site})")
        return False


def _stream_ptr(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _key_bytes(t) -> int:
    es = t.element_size()
    if es not in (4, 8):
        raise TypeError(f"keys must be 4- or 8-byte integers, got {t.dtype}")
    return es


def _require_like(out, numel: int, elem: int, what: str):
    """A caller-supplied output must hold exactly the elements the sort
    writes, of the element width it writes; checked before any launch."""
    if out is None:
        return
    if out.numel() != numel or out.element_size() != elem:
        raise ValueError(f"{what} must hold {numel} elements of {elem} bytes, "
                         f"got {out.numel()} of {out.element_size()}")


def _require_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def temp_bytes(n: int, key_bytes: int, value_bytes: int, begin_bit: int, end_bit: int,
               digit_bits: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().radix_sort_keys_temp_bytes(n, key_bytes, value_bytes, begin_bit,
                                                     end_bit, digit_bits, ctypes.byref(out)),
           "radix_sort_keys_temp_bytes")
    return out.value


def segmented_temp_bytes(rows: int, cols: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().radix_segmented_sort_temp_bytes(rows, cols, ctypes.byref(out)),
           "radix_segmented_sort_temp_bytes")
    return out.value


def _temp(nbytes: int, device, temp=None):
    import torch
    if temp is not None:
        if temp.numel() * temp.element_size() < nbytes:
            raise RadixSortError(RS_ERR_TEMP_TOO_SMALL, "scratch buffer")
        _require_cuda(temp)
        return temp
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _key_type(key_type, kb: int, descending: bool):
    """(type code or None for the unsigned ascending entry points, key bytes)."""
    if key_type is None:
        return (None if not descending else (0 if kb == 4 else 3)), kb
    if key_type not in KEY_TYPES:
        raise ValueError(f"key_type must be one of {sorted(KEY_TYPES)}")
    code, size = KEY_TYPES[key_type]
    if size != kb:
        raise TypeError(f"key_type {key_type} takes {size}-byte keys, got {kb}-byte")
    return (None if code in (0, 3) and not descending else code), kb


def radix_sort_keys(keys, out=None, begin_bit: int = 0, end_bit: int | None = None,
                    digit_bits: int = 8, temp=None, stream=None, key_type=None,
                    descending: bool = False, pass_skipping: bool = False,
                    small_sort: bool = True, lookback_timeout_ns: int = 0):
    """Stable sort of the bits [begin_bit, end_bit) of ``keys``: unsigned and
    ascending by default; ``key_type`` and ``descending`` select the typed
    sort (the bits then belong to the order-preserving transform).  The
    keyword options are those of struct rs_options (include/lsdrs.h)."""
    import torch
    lib = load_library()
    keys = keys.reshape(-1)
    kb = _key_bytes(keys)
    _require_like(out, keys.numel(), kb, "out")
    _require_cuda(keys)
    end_bit = kb * 8 if end_bit is None else end_bit
    if out is None:
        out = torch.empty_like(keys)
    _require_cuda(out)
    n = keys.numel()
    code, _ = _key_type(key_type, kb, descending)
    opts = _options(pass_skipping, False, small_sort, lookback_timeout_ns)
    if opts is not None and code is None:
        code = KEY_TYPES["u32" if kb == 4 else "u64"][0]
    tb = temp_bytes(n, kb, 0, begin_bit, end_bit, digit_bits)
    t = _temp(tb, keys.device, temp)
    tsz = t.numel() * t.element_size()
    with _BoundsGuard(t, stream, "radix_sort_keys"):
        if code is None:
            f = lib.radix_sort_keys_u32 if kb == 4 else lib.radix_sort_keys_u64
            st = f(_ptr(keys), _ptr(out), n, begin_bit, end_bit, digit_bits, _ptr(t), tsz,
                   _stream_ptr(stream))
        else:
            st = lib.radix_sort_keys_typed(code, int(descending), _ptr(keys), _ptr(out), n, begin_bit,
                                           end_bit, digit_bits, _ptr(t), tsz,
                                           ctypes.byref(opts) if opts is not None else None,
                                           _stream_ptr(stream))
        _check(st, "radix_sort_keys")
    return out


def radix_sort_pairs(keys, values, keys_out=None, values_out=None, begin_bit: int = 0,
                     end_bit: int | None = None, digit_bits: int = 8, temp=None, stream=None,
                     key_type=None, descending: bool = False, pass_skipping: bool = False,
                     small_sort: bool = True, lookback_timeout_ns: int = 0):
    """Stable key-value sort: 4-byte ``values`` follow their keys (key order
    and options as for radix_sort_keys)."""
    import torch
    lib = load_library()
    keys = keys.reshape(-1)
    values = values.reshape(-1)
    kb = _key_bytes(keys)
    if values.element_size() != 4 or values.numel() != keys.numel():
        raise ValueError("values must be 4-byte and one per key")
    _require_like(keys_out, keys.numel(), kb, "keys_out")
    _require_like(values_out, keys.numel(), 4, "values_out")
    _require_cuda(keys, values)
    end_bit = kb * 8 if end_bit is None else end_bit
    keys_out = torch.empty_like(keys) if keys_out is None else keys_out
    values_out = torch.empty_like(values) if values_out is None else values_out
    _require_cuda(keys_out, values_out)
    n = keys.numel()
    code, _ = _key_type(key_type, kb, descending)
    opts = _options(pass_skipping, False, small_sort, lookback_timeout_ns)
    if opts is not None and code is None:
        code = KEY_TYPES["u32" if kb == 4 else "u64"][0]
    tb = temp_bytes(n, kb, 4, begin_bit, end_bit, digit_bits)
    t = _temp(tb, keys.device, temp)
    tsz = t.numel() * t.element_size()
    with _BoundsGuard(t, stream, "radix_sort_pairs"):
        if code is None:
            f = lib.radix_sort_pairs_u32 if kb == 4 else lib.radix_sort_pairs_u64
            st = f(_ptr(keys), _ptr(keys_out), _ptr(values), _ptr(values_out), n, begin_bit, end_bit,
                   digit_bits, _ptr(t), tsz, _stream_ptr(stream))
        else:
            st = lib.radix_sort_pairs_typed(code, int(descending), _ptr(keys), _ptr(keys_out),
                                            _ptr(values), _ptr(values_out), n, begin_bit, end_bit,
                                            digit_bits, _ptr(t), tsz,
                                            ctypes.byref(opts) if opts is not None else None,
                                            _stream_ptr(stream))
        _check(st, "radix_sort_pairs")
    return keys_out, values_out


def segmented_sort(x, descending: bool = False, values_out=None, indices_out=None,
                   temp=None, stream=None, tile_offsets: bool = False,
                   pass_skipping: bool = False, small_sort: bool = True,
                   lookback_timeout_ns: int = 0):
    """Row-wise stable sort of a 2-D float16/bfloat16 tensor along the last dim.

    Returns (sorted values, int64 indices), like ``torch.sort(x, dim=-1)``
    with ties in input order, -0 before +0 ascending and NaNs placed by sign
    (negative NaNs first, positive NaNs last; reversed when descending).
    ``tile_offsets`` precomputes each tile's output offsets before every
    pass instead of the look-back; the other options are as for
    radix_sort_keys.
    """
    import torch
    lib = load_library()
    if x.dtype not in (torch.float16, torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("segmented_sort expects float16 or bfloat16 rows")
    if x.dim() != 2:
        raise ValueError("segmented_sort expects a 2-D tensor")
    rows, cols = x.shape
    if values_out is not None and tuple(values_out.shape) != (rows, cols):
        raise ValueError(f"values_out must have shape {(rows, cols)}")
    _require_like(values_out, rows * cols, 2, "values_out")
    if indices_out is not None and (tuple(indices_out.shape) != (rows, cols)
                                    or indices_out.dtype != torch.int64):
        raise ValueError(f"indices_out must be int64 of shape {(rows, cols)}")
    _require_cuda(x)
    kind = RS_BF16 if x.dtype == torch.bfloat16 else RS_F16
    vals = torch.empty_like(x) if values_out is None else values_out
    idx = torch.empty((rows, cols), dtype=torch.int64, device=x.device) \
        if indices_out is None else indices_out
    _require_cuda(vals, idx)
    tb = segmented_temp_bytes(rows, cols)
    t = _temp(tb, x.device, temp)
    opts = _options(pass_skipping, tile_offsets, small_sort, lookback_timeout_ns)
    with _BoundsGuard(t, stream, "radix_segmented_sort_f16"):
        if opts is None:
            st = lib.radix_segmented_sort_f16(_ptr(x), _ptr(vals), _ptr(idx), rows, cols, kind,
                                              int(bool(descending)), _ptr(t),
                                              t.numel() * t.element_size(), _stream_ptr(stream))
        else:
            st = lib.radix_segmented_sort_f16_ex(_ptr(x), _ptr(vals), _ptr(idx), rows, cols, kind,
                                                 int(bool(descending)), _ptr(t),
                                                 t.numel() * t.element_size(), ctypes.byref(opts),
                                                 _stream_ptr(stream))
        _check(st, "radix_segmented_sort_f16")
    return vals, idx


def upfront_histograms(keys, begin_bit: int = 0, end_bit: int | None = None,
                       digit_bits: int = 8, stream=None):
    """(passes, 2**digit_bits) digit counts of every pass and their exclusive scans."""
    import torch
    lib = load_library()
    keys = keys.reshape(-1)
    _require_cuda(keys)
    kb = _key_bytes(keys)
    end_bit = kb * 8 if end_bit is None else end_bit
    passes = -(-(end_bit - begin_bit) // digit_bits) if end_bit > begin_bit else 0
    n = keys.numel()
    tb = temp_bytes(n, kb, 0, begin_bit, end_bit, digit_bits)
    t = _temp(tb, keys.device)
    hist = torch.empty((max(passes, 1), 1 << digit_bits), dtype=torch.int32, device=keys.device)
    bases = torch.empty_like(hist)
    with _BoundsGuard(t, stream, "radix_sort_histograms"):
        _check(lib.radix_sort_histograms(_ptr(keys), kb, n, begin_bit, end_bit, digit_bits,
                                         _ptr(hist), _ptr(bases), _ptr(t),
                                         t.numel() * t.element_size(), _stream_ptr(stream)),
               "radix_sort_histograms")
    return hist[:passes], bases[:passes]


def passes_run(temp, stream=None) -> int:
    """Passes the last sort with this scratch buffer ran (identity passes,
    where every key has the same digit, are skipped).  Synchronises."""
    out = ctypes.c_int(0)
    _check(load_library().radix_sort_passes_run(_ptr(temp), ctypes.byref(out), _stream_ptr(stream)),
           "radix_sort_passes_run")
    return out.value


def device_status(temp, stream=None) -> int:
    """Synchronise and return the device-side status word of the last sort on ``temp``."""
    return int(load_library().radix_sort_device_status(_ptr(temp), _stream_ptr(stream)))


def copy_probe(dst, src, stream=None):
    """Streaming copy of ``src`` into ``dst`` (the bandwidth probe)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() < nbytes:
        raise ValueError("dst is smaller than src")
    _require_cuda(dst, src)
    _check(load_library().rs_copy_probe(_ptr(dst), _ptr(src), nbytes, _stream_ptr(stream)),
           "rs_copy_probe")


def lookback_timeout_probe(timeout_ns: int, stream=None) -> int:
    """Run the bounded look-back wait on a word nothing sets; return its status."""
    import torch
    word = torch.empty(2, dtype=torch.int32, device="cuda")
    res = ctypes.c_int(-1)
    _check(load_library().rs_lookback_timeout_probe(_ptr(word), int(timeout_ns),
                                                    _stream_ptr(stream), ctypes.byref(res)),
           "rs_lookback_timeout_probe")
    return res.value


def profile_enable(on: bool = True):
    _check(load_library().rs_profile_enable(int(bool(on))), "rs_profile_enable")


def profile_read(max_records: int = 1 << 16):
    """[(kernel name, ms, units)] for the launches since the last read."""
    buf = (KernelTime * max_records)()
    n = load_library().rs_profile_read(buf, max_records)
    return [(KERNEL_NAMES.get(buf[i].kernel, str(buf[i].kernel)), buf[i].ms, buf[i].units)
            for i in range(n)]


def launch_count_reset() -> int:
    return int(load_library().rs_launch_count_reset())


def noalloc_status(stream=None) -> int:
    """Synchronise and return the device-side status of the last no-allocation
    sort enqueued on the current device (radix_sort_pairs_u32_noalloc_status)."""
    return int(load_library().radix_sort_pairs_u32_noalloc_status(_stream_ptr(stream)))


def noalloc_timeout_probe(timeout_ns: int, stream=None) -> int:
    """Run the bounded look-back wait on a word of the no-allocation array
    that nothing sets (rs_noalloc_timeout_probe); return its status."""
    res = ctypes.c_int(-1)
    _check(load_library().rs_noalloc_timeout_probe(int(timeout_ns), _stream_ptr(stream),
                                                   ctypes.byref(res)),
           "rs_noalloc_timeout_probe")
    return res.value
