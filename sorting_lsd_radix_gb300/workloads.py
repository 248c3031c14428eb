"""Seeded synthetic key generators shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and shapes them into the key
distributions the sorting pages discuss; it contains none of the sorting
arithmetic (no key encoding, digit, histogram or network code).

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast Splittable
Pseudorandom Number Generators", OOPSLA 2014; the constants of Vigna's public
reference version): draw i of stream ``seed`` is mix(seed + (i + 1) * GAMMA).
Being counter-based, any slice of a stream can be generated independently,
which lets large arrays be produced in parallel chunks with identical results
on any machine.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# Seeds: 0x5EED0000 + 16 * workload index + variant.
SEED_BASE = 0x5EED0000


def seed_for(workload: int, variant: int = 0) -> int:
    return SEED_BASE + 16 * workload + variant


def _mix(z: np.ndarray) -> np.ndarray:
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _draws_chunk(seed: int, start: int, count: int, stride: int, offset: int) -> np.ndarray:
    # counter of draw j = start + i is stride * j + offset (several interleaved sub-streams)
    idx = np.arange(start, start + count, dtype=np.uint64) * np.uint64(stride) + np.uint64(offset + 1)
    with np.errstate(over="ignore"):
        z = idx * GAMMA + np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        return _mix(z)


def splitmix64(seed: int, n: int, stride: int = 1, offset: int = 0) -> np.ndarray:
    """n 64-bit draws: draw i uses counter stride*i + offset of stream seed."""
    out = np.empty(n, dtype=np.uint64)
    if n == 0:
        return out
    starts = list(range(0, n, _CHUNK))

    def work(s):
        c = min(_CHUNK, n - s)
        out[s:s + c] = _draws_chunk(seed, s, c, stride, offset)

    if len(starts) == 1:
        work(0)
    else:
        with _cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out


def _hi32(z: np.ndarray) -> np.ndarray:
    return (z >> np.uint64(32)).astype(np.uint32)


def uniform_u32(n: int, seed: int) -> np.ndarray:
    """i.i.d. uniform over [0, 2^32)."""
    return _hi32(splitmix64(seed, n))


def low_entropy_u32(n: int, seed: int) -> np.ndarray:
    """Bitwise AND of three independent uniform 32-bit draws (each bit set with p = 1/8)."""
    a = _hi32(splitmix64(seed, n, 3, 0))
    a &= _hi32(splitmix64(seed, n, 3, 1))
    a &= _hi32(splitmix64(seed, n, 3, 2))
    return a


def all_equal_u32(n: int, seed: int) -> np.ndarray:
    """Every key equal to one seeded draw."""
    v = _hi32(splitmix64(seed, 1))[0]
    return np.full(n, v, dtype=np.uint32)


def ascending_u32(n: int, seed: int) -> np.ndarray:
    """A non-decreasing sequence built as a running sum of uniform increments.

    Increments are uniform in [0, floor((2^32 - 1) / n)], so the total never
    exceeds 2^32 - 1; zero increments give runs of equal keys.  No sort is used.
    """
    if n == 0:
        return np.zeros(0, dtype=np.uint32)
    step = max((2**32 - 1) // n, 0) + 1
    inc = (splitmix64(seed, n) % np.uint64(step))
    return np.cumsum(inc, dtype=np.uint64).astype(np.uint32)


def descending_u32(n: int, seed: int) -> np.ndarray:
    """The ascending sequence of the same seed, reversed."""
    return np.ascontiguousarray(ascending_u32(n, seed)[::-1])


def uniform_i32(n: int, seed: int) -> np.ndarray:
    """Raw uniform 32-bit draws reinterpreted as signed integers (full signed range)."""
    return uniform_u32(n, seed).view(np.int32)


def uniform_u64(n: int, seed: int) -> np.ndarray:
    return splitmix64(seed, n)


def priority_u64(n: int, seed: int) -> np.ndarray:
    """(16-bit priority uniform in [0, 16)) << 48 | 48-bit uniform field.

    The priority is the top 4 bits of the draw, the field its low 48 bits, so
    bits 52..63 of every key are zero."""
    z = splitmix64(seed, n)
    return ((z >> np.uint64(60)) << np.uint64(48)) | (z & np.uint64((1 << 48) - 1))


def _unit_open(z: np.ndarray) -> np.ndarray:
    # 53-bit uniform in (0, 1]
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def normal_mix_f32(n: int, seed: int, sigma: float = 1e3) -> np.ndarray:
    """f32 N(0, sigma) with 2.5% +0.0, 2.5% -0.0, 0.5% +inf, 0.5% -inf, no NaN.

    The normal draws use the Box-Muller transform in double precision, then
    round to f32; a third draw per element picks the special positions."""
    return _normal_mix(n, seed, sigma, np.float32)


def normal_mix_f64(n: int, seed: int, sigma: float = 1e3) -> np.ndarray:
    """f64 counterpart of normal_mix_f32 (same draws, not rounded to f32)."""
    return _normal_mix(n, seed, sigma, np.float64)


def uniform_i64(n: int, seed: int) -> np.ndarray:
    """Raw uniform 64-bit draws reinterpreted as signed integers (full signed range)."""
    return uniform_u64(n, seed).view(np.int64)


def _normal_mix(n: int, seed: int, sigma: float, dtype) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    if n == 0:
        return out
    starts = list(range(0, n, _CHUNK))

    def work(s):
        c = min(_CHUNK, n - s)
        u1 = _unit_open(_draws_chunk(seed, s, c, 3, 0))
        u2 = _unit_open(_draws_chunk(seed, s, c, 3, 1))
        sel = _hi32(_draws_chunk(seed, s, c, 3, 2)).astype(np.float64) * (1.0 / 4294967296.0)
        x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2) * sigma
        v = x.astype(dtype)
        v[sel < 0.025] = dtype(0.0)
        v[(sel >= 0.025) & (sel < 0.05)] = dtype(-0.0)
        v[(sel >= 0.05) & (sel < 0.055)] = dtype(np.inf)
        v[(sel >= 0.055) & (sel < 0.06)] = dtype(-np.inf)
        out[s:s + c] = v

    if len(starts) == 1:
        work(0)
    else:
        with _cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out


def _to_signed64(x: int) -> int:
    x &= 0xFFFFFFFFFFFFFFFF
    return x - (1 << 64) if x >> 63 else x


def uniform_u32_torch(n: int, seed: int, device, chunk: int = 1 << 26):
    """uniform_u32(n, seed) drawn with torch on `device` (the same SplitMix64 stream, bit for bit),
    returned as an int32 tensor holding the uint32 bit patterns.  For arrays too large to draw on
    the host in reasonable time; int64 arithmetic wraps modulo 2^64, and right shifts are made
    logical by masking."""
    import torch
    out = torch.empty(n, dtype=torch.int32, device=device)
    gamma, m1, m2 = (_to_signed64(int(v)) for v in (GAMMA, _M1, _M2))
    s64 = _to_signed64(seed)

    def lsr(z, k):
        return (z >> k) & ((1 << (64 - k)) - 1)

    for start in range(0, n, chunk):
        c = min(chunk, n - start)
        z = torch.arange(start + 1, start + c + 1, dtype=torch.int64, device=device) * gamma + s64
        z ^= lsr(z, 30)
        z *= m1
        z ^= lsr(z, 27)
        z *= m2
        z ^= lsr(z, 31)
        hi = lsr(z, 32)  # in [0, 2^32)
        out[start:start + c] = torch.where(hi >= (1 << 31), hi - (1 << 32), hi).to(torch.int32)
    return out


def zero_one_patterns(bits: int) -> np.ndarray:
    """Every 0-1 vector of length ``bits`` (2^bits rows, one per pattern), as uint32."""
    codes = np.arange(1 << bits, dtype=np.uint32)
    shifts = np.arange(bits, dtype=np.uint32)
    return ((codes[:, None] >> shifts[None, :]) & np.uint32(1)).astype(np.uint32)


DISTRIBUTIONS_U32 = {
    "uniform": uniform_u32,
    "low_entropy": low_entropy_u32,
    "all_equal": all_equal_u32,
    "sorted": ascending_u32,
    "reverse": descending_u32,
}
