"""Seeded synthetic inputs for the sorts (host side, numpy).

This module holds no sorting arithmetic: it only draws keys.  Both the CUDA
path's tests/benchmark and the CPU oracle take their inputs from here, so the
two sides always see identical bytes.

Random words come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are
Vigna's public ``splitmix64.c``) used in counter mode:

    w(seed, stream, i) = mix64(base(seed, stream) + (i + 1) * GAMMA)
    base(seed, stream) = mix64(seed * 2**32 + stream)

so w(0, 0, .) is exactly the SplitMix64 sequence started from state 0.

Workloads (sizes and value mixes follow the pages' benchmark shapes):
  * uniform u32 keys ``w >> 32`` and small-range keys ``w >> 52`` (< 4096);
  * all-equal, low-entropy (AND of four words), sorted and reverse-sorted u32;
  * uniform u64 keys and skewed u64 keys floor(2**64 * u**8);
  * (rows, cols) fp16/bf16 rows: standard normal by Box-Muller with 1% each
    of +0, -0, +inf, -inf, NaN and 10% duplicated values.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30, _S27, _S31 = np.uint64(30), np.uint64(27), np.uint64(31)

_CHUNK = 1 << 22


def _mix64_inplace(z: np.ndarray) -> np.ndarray:
    z ^= z >> _S30
    z *= _M1
    z ^= z >> _S27
    z *= _M2
    z ^= z >> _S31
    return z


def mix64(x: int) -> int:
    """SplitMix64 finaliser on one Python int (mod 2**64)."""
    m = (1 << 64) - 1
    z = x & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def stream_base(seed: int, stream: int) -> int:
    return mix64(((seed & 0xFFFFFFFF) << 32) | (stream & 0xFFFFFFFF))


def _fill(out: np.ndarray, base: np.uint64, start: int) -> None:
    n = out.size
    with np.errstate(over="ignore"):
        np.add(np.arange(start + 1, start + n + 1, dtype=np.uint64) * GAMMA, base,
               out=out)
    _mix64_inplace(out)


def words(seed: int, stream: int, n: int, start: int = 0,
          threads: int | None = None) -> np.ndarray:
    """w(seed, stream, i) for i in [start, start + n), as uint64."""
    out = np.empty(n, np.uint64)
    base = np.uint64(stream_base(seed, stream))
    if n <= _CHUNK:
        _fill(out, base, start)
        return out
    threads = threads or min(16, os.cpu_count() or 1)
    offs = range(0, n, _CHUNK)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda o: _fill(out[o:o + _CHUNK], base, start + o), offs))
    return out


def word(seed: int, stream: int, i: int) -> int:
    """One word, as a Python int."""
    return mix64(stream_base(seed, stream) + (i + 1) * int(GAMMA))


# ---------------------------------------------------------------- integers

def u32_uniform(n: int, seed: int = 0) -> np.ndarray:
    return (words(seed, 0, n) >> np.uint64(32)).astype(np.uint32)


def u32_small(n: int, seed: int = 0, bits: int = 12) -> np.ndarray:
    """Uniform keys below 2**bits (top bits of the word)."""
    return (words(seed, 0, n) >> np.uint64(64 - bits)).astype(np.uint32)


def u32_all_equal(n: int, seed: int = 0) -> np.ndarray:
    return np.full(n, word(seed, 0, 0) >> 32, np.uint32)


def u32_low_entropy(n: int, seed: int = 0, ands: int = 4) -> np.ndarray:
    """Bitwise AND of ``ands`` uniform words: each bit is set w.p. 2**-ands."""
    acc = words(seed, 0, n) >> np.uint64(32)
    for st in range(1, ands):
        acc &= words(seed, st, n) >> np.uint64(32)
    return acc.astype(np.uint32)


def u32_sorted(n: int, seed: int = 0) -> np.ndarray:
    return np.sort(u32_uniform(n, seed))


def u32_reverse_sorted(n: int, seed: int = 0) -> np.ndarray:
    return np.ascontiguousarray(u32_sorted(n, seed)[::-1])


def u64_uniform(n: int, seed: int = 0) -> np.ndarray:
    return words(seed, 0, n)


def u64_skewed(n: int, seed: int = 0) -> np.ndarray:
    """floor(2**64 * u**8), u = (w >> 11) * 2**-53, u**8 by three IEEE squarings."""
    u = (words(seed, 0, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    u = u * u
    u = u * u
    u = u * u
    x = u * (2.0 ** 64)
    # x < 2**64 always (u < 1); values >= 2**63 need the unsigned conversion.
    hi = x >= 2.0 ** 63
    out = np.empty(n, np.uint64)
    out[~hi] = x[~hi].astype(np.uint64)
    out[hi] = (x[hi] - 2.0 ** 63).astype(np.uint64) + np.uint64(1 << 63)
    return out


def index_payload(n: int) -> np.ndarray:
    return np.arange(n, dtype=np.uint32)


U32_DISTRIBUTIONS = {
    "uniform": u32_uniform,
    "all_equal": u32_all_equal,
    "low_entropy": u32_low_entropy,
    "sorted": u32_sorted,
    "reverse_sorted": u32_reverse_sorted,
}

U64_DISTRIBUTIONS = {
    "uniform": u64_uniform,
    "skewed": u64_skewed,
}

# ------------------------------------------------------------ 16-bit floats

F16_PZERO, F16_NZERO = 0x0000, 0x8000
F16_PINF, F16_NINF = 0x7C00, 0xFC00
F16_PNAN, F16_NNAN = 0x7E00, 0xFE00
BF16_PINF, BF16_NINF = 0x7F80, 0xFF80
BF16_PNAN, BF16_NNAN = 0x7FC0, 0xFFC0


def double_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite doubles to bfloat16 bit patterns, nearest-even, in one step.

    Handles zero and the normal range of bfloat16 (the Box-Muller samples);
    anything outside it goes through float32 (not reached by these workloads).
    """
    x = np.asarray(x, np.float64)
    bits = x.view(np.uint64)
    sign = (bits >> np.uint64(63)).astype(np.uint32)
    exp = ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64) - 1023 + 127
    mant = bits & np.uint64((1 << 52) - 1)
    keep = (mant >> np.uint64(45)).astype(np.uint32)           # top 7 bits
    rnd = ((mant >> np.uint64(44)) & np.uint64(1)).astype(np.uint32)
    sticky = (mant & np.uint64((1 << 44) - 1)) != 0
    inc = (rnd == 1) & (sticky | ((keep & 1) == 1))
    mag = (np.clip(exp, 0, 255).astype(np.uint32) << 7) + keep + inc.astype(np.uint32)
    out = ((sign << 15) | mag).astype(np.uint16)
    normal = (exp >= 1) & (exp <= 254)
    if not normal.all():
        f = x[~normal].astype(np.float32).view(np.uint32)
        r = ((f >> 16) & 1) + 0x7FFF
        out[~normal] = ((f + r) >> 16).astype(np.uint16)
        zero = x == 0.0
        out[zero] = (sign[zero] << 15).astype(np.uint16)
    return out


def _rows16_block(out: np.ndarray, r0: int, rows: int, cols: int, kind: str, seed: int,
                  specials: bool) -> None:
    start, n = r0 * cols, rows * cols
    sh = np.uint64(11)
    u1 = ((words(seed, 0, n, start, 1) >> sh).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (words(seed, 1, n, start, 1) >> sh).astype(np.float64) * (2.0 ** -53)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    del u1, u2
    if kind == "f16":
        base = z.astype(np.float16).view(np.uint16)
        pinf, ninf, pnan, nnan = F16_PINF, F16_NINF, F16_PNAN, F16_NNAN
    else:
        base = double_to_bf16_bits(z)
        pinf, ninf, pnan, nnan = BF16_PINF, BF16_NINF, BF16_PNAN, BF16_NNAN
    del z
    base = base.reshape(rows, cols)
    if not specials:
        out[...] = base
        return
    blk = base.copy()
    u = (words(seed, 2, n, start, 1) >> sh).astype(np.float64).reshape(rows, cols) * (2.0 ** -53)
    nan_sign = (words(seed, 3, n, start, 1) & np.uint64(1)).reshape(rows, cols).astype(bool)
    src_col = (words(seed, 4, n, start, 1) % np.uint64(cols)).astype(np.int64).reshape(rows, cols)
    blk[u < 0.01] = F16_PZERO
    blk[(u >= 0.01) & (u < 0.02)] = F16_NZERO
    blk[(u >= 0.02) & (u < 0.03)] = pinf
    blk[(u >= 0.03) & (u < 0.04)] = ninf
    nan = (u >= 0.04) & (u < 0.05)
    blk[nan & ~nan_sign] = pnan
    blk[nan & nan_sign] = nnan
    dup = (u >= 0.05) & (u < 0.15)
    r_idx = np.broadcast_to(np.arange(rows)[:, None], (rows, cols))
    blk[dup] = base[r_idx[dup], src_col[dup]]
    out[...] = blk


def rows16(rows: int, cols: int, kind: str = "f16", seed: int = 0,
           specials: bool = True, threads: int | None = None) -> np.ndarray:
    """(rows, cols) uint16 bit patterns of fp16 ("f16") or bf16 ("bf16") values.

    Base value: standard normal by Box-Muller from two 53-bit uniforms
    (streams 0 and 1), rounded to the format nearest-even.  With ``specials``:
    for u = w(seed, 2, i) * 2**-64, [0,.01) +0, [.01,.02) -0, [.02,.03) +inf,
    [.03,.04) -inf, [.04,.05) NaN (sign = bit 0 of w(seed, 3, i)) and
    [.05,.15) a copy of the base value at column w(seed, 4, i) mod cols of the
    same row.  i is the flat row-major index.
    """
    if kind not in ("f16", "bf16"):
        raise ValueError("kind must be 'f16' or 'bf16'")
    out = np.empty((rows, cols), np.uint16)
    if rows == 0 or cols == 0:
        return out
    per = max(1, (1 << 20) // max(cols, 1))
    blocks = [(r, min(per, rows - r)) for r in range(0, rows, per)]
    threads = threads or min(16, os.cpu_count() or 1)
    if len(blocks) == 1:
        _rows16_block(out, 0, rows, cols, kind, seed, specials)
        return out
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda b: _rows16_block(out[b[0]:b[0] + b[1]], b[0], b[1], cols, kind,
                                            seed, specials), blocks))
    return out
