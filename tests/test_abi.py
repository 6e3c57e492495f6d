"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments on the host before anything is enqueued (no GPU use)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "lsdrs.h")


@pytest.fixture(scope="module")
def lib():
    from lsd_radix_sort_gb300 import build
    build.build()
    import lsd_radix_sort_gb300 as rs
    return rs.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    import lsd_radix_sort_gb300 as rs
    assert set(rs.EXPORTED_SYMBOLS) == set(names), (set(rs.EXPORTED_SYMBOLS) ^ set(names))


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.rs_status_string(0) == b"RS_OK"
    assert lib.rs_status_string(4) == b"RS_ERR_LOOKBACK_TIMEOUT"
    assert lib.rs_status_string(99) == b"RS_UNKNOWN"


def test_temp_bytes_query(lib):
    out = ctypes.c_size_t(0)
    assert lib.radix_sort_keys_temp_bytes(1 << 20, 4, 4, 0, 32, 8, ctypes.byref(out)) == 0
    n = 1 << 20
    assert out.value >= n * 8            # alternate keys + payloads
    small = ctypes.c_size_t(0)
    assert lib.radix_sort_keys_temp_bytes(1 << 20, 4, 0, 0, 32, 8, ctypes.byref(small)) == 0
    assert small.value < out.value
    assert lib.radix_segmented_sort_temp_bytes(1024, 65536, ctypes.byref(out)) == 0
    assert lib.radix_segmented_sort_temp_bytes(1 << 40, 1 << 10, ctypes.byref(out)) == 1
    assert out.value >= 1024 * 65536 * 6  # alternate keys + int32 indices
    assert lib.radix_sort_keys_temp_bytes(0, 4, 0, 0, 32, 8, ctypes.byref(out)) == 0
    # flat sorts of 2^30 keys and more are accepted (segmented look-back), up
    # to 2^32 - 1; a row of a row-wise sort stays below 2^30
    assert lib.radix_sort_keys_temp_bytes((1 << 32) - 1, 4, 4, 0, 32, 8, ctypes.byref(out)) == 0
    assert out.value >= ((1 << 32) - 1) * 8
    assert lib.radix_segmented_sort_temp_bytes(1, 1 << 30, ctypes.byref(out)) == 1
    assert lib.radix_segmented_sort_temp_bytes(2, (1 << 30) - 1, ctypes.byref(out)) == 0


@pytest.mark.parametrize("args", [
    (1 << 10, 3, 0, 0, 32, 8),       # key bytes
    (1 << 10, 4, 2, 0, 32, 8),       # value bytes
    (1 << 10, 4, 0, 0, 33, 8),       # end bit past the key
    (1 << 10, 4, 0, 8, 8, 8),        # empty bit range
    (1 << 10, 4, 0, -1, 8, 8),
    (1 << 10, 4, 0, 0, 32, 0),       # digit width
    (1 << 10, 4, 0, 0, 32, 9),
    (1 << 32, 4, 0, 0, 32, 8),       # beyond RS_MAX_KEYS
])
def test_temp_bytes_rejects(lib, args):
    out = ctypes.c_size_t(0)
    assert lib.radix_sort_keys_temp_bytes(*args, ctypes.byref(out)) == 1


def test_sort_calls_validate_before_launch(lib):
    """Every one of these returns on the host; the pointers are never touched."""
    bogus = ctypes.c_void_p(0x1000)
    temp = ctypes.c_void_p(0x100000)
    big = 1 << 40
    # bad digit width / bit range
    assert lib.radix_sort_keys_u32(bogus, bogus, 100, 0, 32, 0, temp, big, None) == 1
    assert lib.radix_sort_keys_u64(bogus, bogus, 100, 0, 65, 8, temp, big, None) == 1
    assert lib.radix_sort_pairs_u32(bogus, bogus, bogus, bogus, 100, 5, 5, 8, temp, big, None) == 1
    # too many keys
    assert lib.radix_sort_keys_u32(bogus, bogus, 1 << 32, 0, 32, 8, temp, big, None) == 1
    # temp too small
    assert lib.radix_sort_keys_u32(bogus, ctypes.c_void_p(0x90000000), 100, 0, 32, 8, temp, 16,
                                   None) == 2
    # missing temp / null pointers
    assert lib.radix_sort_keys_u32(bogus, bogus, 100, 0, 32, 8, None, big, None) == 1
    assert lib.radix_sort_pairs_u32(bogus, ctypes.c_void_p(0x90000000), None, None, 100, 0, 32, 8,
                                    temp, big, None) == 1
    # partially overlapping input and output
    assert lib.radix_sort_keys_u32(ctypes.c_void_p(0x20000000), ctypes.c_void_p(0x20000004), 100,
                                   0, 32, 8, temp, big, None) == 1
    # misaligned temp
    assert lib.radix_sort_keys_u32(bogus, ctypes.c_void_p(0x90000000), 100, 0, 32, 8,
                                   ctypes.c_void_p(0x100004), big, None) == 1
    # n == 0 is a no-op
    assert lib.radix_sort_keys_u32(None, None, 0, 0, 32, 8, None, 0, None) == 0
    # row-wise sort: bad kind / descending flag / negative shape
    assert lib.radix_segmented_sort_f16(bogus, bogus, bogus, 2, 2, 7, 0, temp, big, None) == 1
    assert lib.radix_segmented_sort_f16(bogus, bogus, bogus, 2, 2, 0, 2, temp, big, None) == 1
    assert lib.radix_segmented_sort_f16(bogus, bogus, bogus, -1, 2, 0, 0, temp, big, None) == 1
    assert lib.radix_segmented_sort_f16(bogus, bogus, bogus, 0, 5, 0, 0, temp, big, None) == 0
    # more rows than tile ids (and rows * cols past any buffer): refused
    assert lib.radix_segmented_sort_f16(bogus, bogus, bogus, 1 << 40, 1 << 20, 0, 0, temp, big,
                                        None) == 1
    assert lib.radix_segmented_sort_f16(bogus, bogus, bogus, 1 << 62, 4, 0, 0, temp, big,
                                        None) == 1
    # typed sorts: unknown key type, bad descending flag, bad bit range, n == 0
    assert lib.radix_sort_keys_typed(9, 0, bogus, bogus, 100, 0, 32, 8, temp, big, None,
                                     None) == 1
    assert lib.radix_sort_keys_typed(-1, 0, bogus, bogus, 100, 0, 32, 8, temp, big, None,
                                     None) == 1
    assert lib.radix_sort_keys_typed(1, 2, bogus, bogus, 100, 0, 32, 8, temp, big, None,
                                     None) == 1
    assert lib.radix_sort_keys_typed(2, 0, bogus, bogus, 100, 0, 33, 8, temp, big, None,
                                     None) == 1
    assert lib.radix_sort_pairs_typed(5, 1, bogus, bogus, bogus, bogus, 100, 0, 65, 8, temp, big,
                                      None, None) == 1
    assert lib.radix_sort_pairs_typed(4, 0, bogus, bogus, None, None, 100, 0, 64, 8, temp, big,
                                      None, None) == 1
    assert lib.radix_sort_keys_typed(2, 1, None, None, 0, 0, 32, 8, None, 0, None, None) == 0
    # histograms: bad key width
    assert lib.radix_sort_histograms(bogus, 2, 100, 0, 16, 8, bogus, bogus, temp, big, None) == 1
    # copy probe: misaligned sizes
    assert lib.rs_copy_probe(bogus, temp, 15, None) == 1
    # look-back probe: wait limit above 60 s
    assert lib.rs_lookback_timeout_probe(bogus, 61_000_000_000, None, ctypes.byref(
        ctypes.c_int(0))) == 1


def test_options_validated_before_launch(lib):
    """Per-call options: unknown flag bits and a wait limit above 60 s are
    refused on the host; the pointers are never touched."""
    import lsd_radix_sort_gb300 as rs
    bogus = ctypes.c_void_p(0x1000)
    out = ctypes.c_void_p(0x90000000)
    temp = ctypes.c_void_p(0x100000)
    big = 1 << 40
    n = 100_000
    for opts in (rs.Options(0x8, 0), rs.Options(0, 61_000_000_000)):
        assert lib.radix_sort_pairs_typed(0, 0, bogus, out, ctypes.c_void_p(0x50000000),
                                          ctypes.c_void_p(0x60000000), n, 0, 32, 8, temp, big,
                                          ctypes.byref(opts), None) == 1
    assert lib.radix_sort_keys_typed(1, 0, bogus, out, n, 0, 32, 8, temp, big,
                                     ctypes.byref(rs.Options(0x10, 0)), None) == 1
    assert lib.radix_segmented_sort_f16_ex(bogus, out, ctypes.c_void_p(0x50000000), 2, 100, 0, 0,
                                           temp, big, ctypes.byref(rs.Options(0x80, 0)),
                                           None) == 1


def test_temp_bytes_widen_lookback_words_from_2p30(lib):
    """From 2^30 keys a flat sort's look-back words are 64-bit: the scratch
    grows by the status arrays' second half, beyond the ping-pong buffers."""
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    n = (1 << 30) - 1
    assert lib.radix_sort_keys_temp_bytes(n, 4, 4, 0, 32, 8, ctypes.byref(a)) == 0
    assert lib.radix_sort_keys_temp_bytes(n + 1, 4, 4, 0, 32, 8, ctypes.byref(b)) == 0
    tiles = -(-(n + 1) // 5888)
    assert b.value - a.value >= 2 * tiles * 256 * 4  # two status arrays, 4 more bytes a word


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    import lsd_radix_sort_gb300 as rs
    monkeypatch.setattr(rs, "_lib", None)
    monkeypatch.setattr(rs._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        rs.load_library()
