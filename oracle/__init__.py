"""Sorting oracle: numpy front end of the plain single-threaded C reference.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  Nothing here imports, loads or shares
code with the CUDA library; ``oracle.c`` restates the pages' algorithms on its
own (serial LSD counting sort, recursive bitonic network, key encodings).

Key kinds follow numpy dtypes: uint32, int32, float32, uint64, int64 and float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

KIND_U32, KIND_I32, KIND_F32, KIND_U64, KIND_I64, KIND_F64 = 0, 1, 2, 3, 4, 5
_KINDS = {
    np.dtype(np.uint32): KIND_U32,
    np.dtype(np.int32): KIND_I32,
    np.dtype(np.float32): KIND_F32,
    np.dtype(np.uint64): KIND_U64,
    np.dtype(np.int64): KIND_I64,
    np.dtype(np.float64): KIND_F64,
}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with the host C compiler."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(os.path.join(_HERE, "oracle.h")))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-Wall", "-Wextra",
                               _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    vp, sz, i, u64p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)
    lib.orc_key_transform.restype = ctypes.c_uint64
    lib.orc_key_transform.argtypes = [i, ctypes.c_uint64, i]
    lib.orc_key_inverse.restype = ctypes.c_uint64
    lib.orc_key_inverse.argtypes = [i, ctypes.c_uint64, i]
    lib.orc_num_passes.argtypes = [i, i]
    lib.orc_key_transform_array.argtypes = [i, vp, sz, i, vp]
    lib.orc_key_inverse_array.argtypes = [i, vp, sz, i, vp]
    lib.orc_digit_histograms.argtypes = [i, vp, sz, i, i, i, vp]
    lib.orc_lsd_radix_sort.argtypes = [i, vp, vp, sz, i, i, i, vp, vp]
    lib.orc_bitonic_sort.argtypes = [i, vp, sz, i, vp, u64p, u64p]
    lib.orc_segmented_sort.argtypes = [i, vp, sz, sz, i, vp]
    lib.orc_bitonic_split_u32.argtypes = [vp, sz, i]
    lib.orc_bitonic_merge_u32.argtypes = [vp, sz, i]
    _lib = lib
    return lib


def _kind(a: np.ndarray) -> int:
    try:
        return _KINDS[a.dtype]
    except KeyError:
        raise TypeError(f"unsupported key dtype {a.dtype}") from None


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a.size else ctypes.c_void_p(0)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def key_bits(dtype) -> int:
    return np.dtype(dtype).itemsize * 8


def transform(kind: int, raw: int, descending: bool = False) -> int:
    """Order-preserving code of one raw key bit pattern."""
    return int(_load().orc_key_transform(kind, int(raw), int(bool(descending))))


def inverse(kind: int, code: int, descending: bool = False) -> int:
    return int(_load().orc_key_inverse(kind, int(code), int(bool(descending))))


def transform_array(keys: np.ndarray, descending: bool = False) -> np.ndarray:
    """Order-preserving codes (uint64) of every key."""
    keys = np.ascontiguousarray(keys)
    codes = np.empty(keys.size, dtype=np.uint64)
    _check(_load().orc_key_transform_array(_kind(keys), _ptr(keys), keys.size, int(bool(descending)),
                                           _ptr(codes)), "transform_array")
    return codes


def inverse_array(codes: np.ndarray, dtype, descending: bool = False) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint64)
    out = np.empty(codes.size, dtype=dtype)
    _check(_load().orc_key_inverse_array(_kind(out), _ptr(codes), codes.size, int(bool(descending)),
                                         _ptr(out)), "inverse_array")
    return out


def num_passes(begin_bit: int, end_bit: int) -> int:
    return int(_load().orc_num_passes(begin_bit, end_bit))


def digit_histograms(keys: np.ndarray, begin_bit: int = 0, end_bit: int | None = None,
                     descending: bool = False) -> np.ndarray:
    """[passes, 256] digit counts of the transformed keys."""
    keys = np.ascontiguousarray(keys)
    if end_bit is None:
        end_bit = key_bits(keys.dtype)
    hist = np.zeros((max(num_passes(begin_bit, end_bit), 1), 256), dtype=np.uint64)
    _check(_load().orc_digit_histograms(_kind(keys), _ptr(keys), keys.size, begin_bit, end_bit,
                                        int(bool(descending)), _ptr(hist)), "digit_histograms")
    return hist[: num_passes(begin_bit, end_bit)]


def sort_keys(keys: np.ndarray, begin_bit: int = 0, end_bit: int | None = None,
              descending: bool = False) -> np.ndarray:
    """Stable LSD radix sort of keys by bits [begin_bit, end_bit) of their code."""
    keys = np.ascontiguousarray(keys)
    if end_bit is None:
        end_bit = key_bits(keys.dtype)
    out = np.empty_like(keys)
    _check(_load().orc_lsd_radix_sort(_kind(keys), _ptr(keys), None, keys.size, begin_bit, end_bit,
                                      int(bool(descending)), _ptr(out), None), "sort_keys")
    return out


def sort_pairs(keys: np.ndarray, vals: np.ndarray, begin_bit: int = 0, end_bit: int | None = None,
               descending: bool = False):
    """Stable LSD radix sort of (key, uint32 value) pairs."""
    keys = np.ascontiguousarray(keys)
    vals = np.ascontiguousarray(vals, dtype=np.uint32)
    if vals.size != keys.size:
        raise ValueError("keys and values differ in length")
    if end_bit is None:
        end_bit = key_bits(keys.dtype)
    ko = np.empty_like(keys)
    vo = np.empty_like(vals)
    _check(_load().orc_lsd_radix_sort(_kind(keys), _ptr(keys), _ptr(vals), keys.size, begin_bit,
                                      end_bit, int(bool(descending)), _ptr(ko), _ptr(vo)), "sort_pairs")
    return ko, vo


def bitonic_sort(keys: np.ndarray, descending: bool = False, count: bool = False):
    """Recursive bitonic network sort of one array (padded to a power of two).

    With count=True also returns (comparators executed, network depth)."""
    keys = np.ascontiguousarray(keys)
    out = np.empty_like(keys)
    comps = ctypes.c_uint64(0)
    depth = ctypes.c_uint64(0)
    _check(_load().orc_bitonic_sort(_kind(keys), _ptr(keys), keys.size, int(bool(descending)), _ptr(out),
                                    ctypes.byref(comps) if count else None,
                                    ctypes.byref(depth) if count else None), "bitonic_sort")
    if count:
        return out, int(comps.value), int(depth.value)
    return out


def segmented_sort(keys: np.ndarray, num_segments: int, segment_len: int,
                   descending: bool = False) -> np.ndarray:
    keys = np.ascontiguousarray(keys)
    if keys.size != num_segments * segment_len:
        raise ValueError("keys.size != num_segments * segment_len")
    out = np.empty_like(keys)
    _check(_load().orc_segmented_sort(_kind(keys), _ptr(keys), num_segments, segment_len,
                                      int(bool(descending)), _ptr(out)), "segmented_sort")
    return out


def bitonic_split(a: np.ndarray, up: bool = True) -> np.ndarray:
    a = np.array(a, dtype=np.uint32)
    _check(_load().orc_bitonic_split_u32(_ptr(a), a.size, int(bool(up))), "bitonic_split")
    return a


def bitonic_merge(a: np.ndarray, up: bool = True) -> np.ndarray:
    a = np.array(a, dtype=np.uint32)
    _check(_load().orc_bitonic_merge_u32(_ptr(a), a.size, int(bool(up))), "bitonic_merge")
    return a
