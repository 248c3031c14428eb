"""Python binding of the gbsort C ABI (include/gbsort.h).

Argument marshalling only: every function forwards torch tensors' device
pointers, sizes and the current CUDA stream to the entry point of the same
name in libgbsort.so; all sorting work runs in that library's kernels.  The
work buffer is a torch uint8 tensor that the caller may pass in and reuse
(it is allocated here, never inside the library).

The library is loaded on first use; if it is missing the call raises, so no
computation can silently happen elsewhere.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbsort.so")

GBS_OK, GBS_ERR_INVALID_ARG, GBS_ERR_TEMP_TOO_SMALL, GBS_ERR_UNSUPPORTED, GBS_ERR_CUDA, GBS_ERR_TIMEOUT = range(6)
GBS_U32, GBS_I32, GBS_F32, GBS_U64, GBS_I64, GBS_F64 = range(6)
GBS_MAX_RADIX_KEYS = (1 << 32) - 1
GBS_MAX_SEGMENT_LEN = 16384

_DTYPE_KIND = {
    torch.uint32: GBS_U32,
    torch.int32: GBS_I32,
    torch.float32: GBS_F32,
    torch.uint64: GBS_U64,
    torch.int64: GBS_I64,
    torch.float64: GBS_F64,
}
_KIND_BYTES = {GBS_U32: 4, GBS_I32: 4, GBS_F32: 4, GBS_U64: 8, GBS_I64: 8, GBS_F64: 8}

# every symbol the headers declare
EXPORTS = ("gbs_sort_keys", "gbs_sort_pairs", "gbs_segmented_sort", "gbs_digit_histograms", "gbs_get_status",
           "gbs_status_string", "gbs_version", "gbs_debug_set_lookback_fault", "gbs_debug_last_launch_count",
           "gbs_debug_radix_tile_keys", "gbs_debug_set_timing_events", "gbs_sort_keys_noalloc",
           "gbs_sort_keys_host", "gbs_segmented_sort_offsets", "gbs_sort_pairs64", "gbs_get_status_noalloc",
           "gbs_sort_keys_msd_bitonic", "gbs_debug_set_radix_bits", "gbs_sort_keys_host_batch")
GBS_NOALLOC_MAX_KEYS = 1 << 20


class GbsError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


_lib = None


def load(path: str | None = None):
    """Loads libgbsort.so (built by sorting_lsd_radix_gb300.build) and declares the prototypes."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"gbsort CUDA library not built: {p} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    vp, sz, i, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    szp = ctypes.POINTER(ctypes.c_size_t)
    lib.gbs_sort_keys.argtypes = [vp, szp, i, vp, vp, sz, i, i, i, vp]
    lib.gbs_sort_keys.restype = i
    lib.gbs_sort_keys_host.argtypes = [vp, szp, i, vp, vp, sz, i, i, i, vp]
    lib.gbs_sort_keys_host_batch.restype = i
    lib.gbs_sort_keys_host_batch.argtypes = [vp, szp, i, ctypes.POINTER(vp), ctypes.POINTER(vp), szp, sz, i, i, i,
                                             vp]
    lib.gbs_sort_keys_host.restype = i
    lib.gbs_sort_pairs.argtypes = [vp, szp, i, vp, vp, vp, vp, sz, i, i, i, vp]
    lib.gbs_sort_pairs64.argtypes = [vp, szp, i, vp, vp, vp, vp, sz, i, i, i, vp]
    lib.gbs_sort_pairs64.restype = i
    lib.gbs_sort_pairs.restype = i
    lib.gbs_segmented_sort_offsets.argtypes = [vp, szp, i, vp, vp, sz, vp, i, vp]
    lib.gbs_segmented_sort_offsets.restype = i
    lib.gbs_segmented_sort.argtypes = [vp, szp, i, vp, vp, sz, sz, i, vp]
    lib.gbs_segmented_sort.restype = i
    lib.gbs_digit_histograms.argtypes = [vp, szp, i, vp, sz, i, i, i, vp, vp]
    lib.gbs_digit_histograms.restype = i
    lib.gbs_sort_keys_noalloc.argtypes = [i, vp, vp, sz, i, i, i, vp]
    lib.gbs_sort_keys_noalloc.restype = i
    lib.gbs_sort_keys_msd_bitonic.argtypes = [vp, szp, i, vp, vp, sz, i, vp]
    lib.gbs_sort_keys_msd_bitonic.restype = i
    lib.gbs_debug_set_radix_bits.argtypes = [i]
    lib.gbs_debug_set_radix_bits.restype = None
    lib.gbs_get_status_noalloc.argtypes = [vp]
    lib.gbs_get_status_noalloc.restype = i
    lib.gbs_get_status.argtypes = [vp, sz, vp]
    lib.gbs_get_status.restype = i
    lib.gbs_status_string.argtypes = [i]
    lib.gbs_status_string.restype = ctypes.c_char_p
    lib.gbs_version.argtypes = []
    lib.gbs_version.restype = ctypes.c_char_p
    lib.gbs_debug_set_lookback_fault.argtypes = [i, u32, u32]
    lib.gbs_debug_set_lookback_fault.restype = None
    lib.gbs_debug_last_launch_count.argtypes = []
    lib.gbs_debug_last_launch_count.restype = i
    lib.gbs_debug_radix_tile_keys.argtypes = [i, i]
    lib.gbs_debug_radix_tile_keys.restype = sz
    lib.gbs_debug_set_timing_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i]
    lib.gbs_debug_set_timing_events.restype = None
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().gbs_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


def gbs_version() -> str:
    return load().gbs_version().decode()


def _kind(t: torch.Tensor, key_type: int | None) -> int:
    if key_type is not None:
        if _KIND_BYTES[key_type] != t.element_size():
            raise ValueError("key_type does not match the tensor's element size")
        return key_type
    try:
        return _DTYPE_KIND[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported key dtype {t.dtype}; pass key_type for a reinterpreting view") from None


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr() if t is not None and t.numel() else 0)


def _check_tensor(t: torch.Tensor, n: int, what: str):
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.numel() != n:
        raise ValueError(f"{what} must hold {n} elements")


def _run(fn, args_after_temp, temp: torch.Tensor | None, what: str) -> torch.Tensor:
    """Work-buffer protocol: with a work buffer, run at once; without one, or if it is too small
    (GBS_ERR_TEMP_TOO_SMALL, nothing launched), query the size, allocate with torch and run."""
    if temp is not None:
        have = ctypes.c_size_t(temp.numel())
        st = fn(_ptr(temp), ctypes.byref(have), *args_after_temp)
        if st == GBS_OK:
            return temp
        if st != GBS_ERR_TEMP_TOO_SMALL:
            raise GbsError(st, what)
    need = ctypes.c_size_t(0)
    st = fn(None, ctypes.byref(need), *args_after_temp)
    if st != GBS_OK:
        raise GbsError(st, what)
    temp = torch.empty(max(need.value, 256), dtype=torch.uint8, device="cuda")
    have = ctypes.c_size_t(temp.numel())
    st = fn(_ptr(temp), ctypes.byref(have), *args_after_temp)
    if st != GBS_OK:
        raise GbsError(st, what)
    return temp


def temp_bytes(fn_name: str, *args) -> int:
    """Work-buffer size a call with these C-level arguments needs (no launch)."""
    need = ctypes.c_size_t(0)
    st = getattr(load(), fn_name)(None, ctypes.byref(need), *args)
    if st != GBS_OK:
        raise GbsError(st, fn_name)
    return need.value


def gbs_sort_keys(keys_in: torch.Tensor, keys_out: torch.Tensor | None = None, begin_bit: int = 0,
                  end_bit: int | None = None, descending: bool = False, temp: torch.Tensor | None = None,
                  key_type: int | None = None, stream=None, return_temp: bool = False):
    """Stable LSD radix sort of a CUDA tensor of keys by bits [begin_bit, end_bit) of their code.

    keys_out may be keys_in (in place); None allocates a new tensor."""
    kind = _kind(keys_in, key_type)
    n = keys_in.numel()
    _check_tensor(keys_in, n, "keys_in")
    if keys_out is None:
        keys_out = torch.empty_like(keys_in)
    _check_tensor(keys_out, n, "keys_out")
    if end_bit is None:
        end_bit = 8 * _KIND_BYTES[kind]
    args = (kind, _ptr(keys_in), _ptr(keys_out), n, begin_bit, end_bit, int(bool(descending)), _stream(stream))
    temp = _run(load().gbs_sort_keys, args, temp, "gbs_sort_keys")
    return (keys_out, temp) if return_temp else keys_out


def gbs_sort_keys_msd_bitonic(keys_in: torch.Tensor, keys_out: torch.Tensor | None = None,
                              descending: bool = False, temp: torch.Tensor | None = None,
                              key_type: int | None = None, stream=None, return_temp: bool = False):
    """Full-width key sort by MSD radix passes over the top 16 bits, then a bitonic sort of every
    bucket (the pages' hybrid; synchronises the stream once)."""
    kind = _kind(keys_in, key_type)
    n = keys_in.numel()
    _check_tensor(keys_in, n, "keys_in")
    if keys_out is None:
        keys_out = torch.empty_like(keys_in)
    _check_tensor(keys_out, n, "keys_out")
    args = (kind, _ptr(keys_in), _ptr(keys_out), n, int(bool(descending)), _stream(stream))
    temp = _run(load().gbs_sort_keys_msd_bitonic, args, temp, "gbs_sort_keys_msd_bitonic")
    return (keys_out, temp) if return_temp else keys_out


def gbs_sort_keys_host(keys_in: torch.Tensor, keys_out: torch.Tensor | None = None, begin_bit: int = 0,
                       end_bit: int | None = None, descending: bool = False, temp: torch.Tensor | None = None,
                       key_type: int | None = None, stream=None, return_temp: bool = False):
    """gbs_sort_keys on a CPU tensor: copy to the device, sort, copy back into keys_out (a CPU tensor;
    may be keys_in; None allocates one, page-locked when keys_in is).  Asynchronous on the stream:
    synchronise it before reading keys_out.  temp is the device work buffer (torch uint8)."""
    kind = _kind(keys_in, key_type)
    n = keys_in.numel()
    if keys_in.is_cuda or not keys_in.is_contiguous():
        raise ValueError("keys_in must be a contiguous CPU tensor")
    if keys_out is None:
        keys_out = torch.empty_like(keys_in, pin_memory=keys_in.is_pinned())
    if keys_out.is_cuda or not keys_out.is_contiguous() or keys_out.numel() != n:
        raise ValueError(f"keys_out must be a contiguous CPU tensor of {n} elements")
    if end_bit is None:
        end_bit = 8 * _KIND_BYTES[kind]
    args = (kind, _ptr(keys_in), _ptr(keys_out), n, begin_bit, end_bit, int(bool(descending)), _stream(stream))
    temp = _run(load().gbs_sort_keys_host, args, temp, "gbs_sort_keys_host")
    return (keys_out, temp) if return_temp else keys_out


def gbs_sort_keys_host_batch(keys_in: list, keys_out: list | None = None, begin_bit: int = 0,
                             end_bit: int | None = None, descending: bool = False, temp: torch.Tensor | None = None,
                             key_type: int | None = None, stream=None, return_temp: bool = False):
    """gbs_sort_keys_host on a list of CPU tensors of one dtype, with the copies of neighbouring arrays
    overlapped (see the C entry point).  keys_out: a list of CPU tensors of the same sizes (an entry may be
    the matching keys_in), or None to allocate them (page-locked when the inputs are).  Asynchronous on the
    stream: synchronise it before reading the outputs."""
    kind = _kind(keys_in[0], key_type) if keys_in else (GBS_U32 if key_type is None else key_type)
    for t in keys_in:
        if t.is_cuda or not t.is_contiguous() or t.dtype != keys_in[0].dtype:
            raise ValueError("keys_in must be contiguous CPU tensors of one dtype")
    if keys_out is None:
        keys_out = [torch.empty_like(t, pin_memory=t.is_pinned()) for t in keys_in]
    if len(keys_out) != len(keys_in):
        raise ValueError("keys_out must hold one tensor per input")
    for t, o in zip(keys_in, keys_out):
        if o.is_cuda or not o.is_contiguous() or o.numel() != t.numel() or o.dtype != t.dtype:
            raise ValueError("each keys_out entry must be a contiguous CPU tensor like its input")
    if end_bit is None:
        end_bit = 8 * _KIND_BYTES[kind]
    count = len(keys_in)
    ins = (ctypes.c_void_p * max(count, 1))(*[_ptr(t) for t in keys_in])
    outs = (ctypes.c_void_p * max(count, 1))(*[_ptr(t) for t in keys_out])
    ns = (ctypes.c_size_t * max(count, 1))(*[t.numel() for t in keys_in])
    args = (kind, ins, outs, ns, count, begin_bit, end_bit, int(bool(descending)), _stream(stream))
    temp = _run(load().gbs_sort_keys_host_batch, args, temp, "gbs_sort_keys_host_batch")
    return (keys_out, temp) if return_temp else keys_out


def gbs_sort_pairs(keys_in: torch.Tensor, vals_in: torch.Tensor, keys_out: torch.Tensor | None = None,
                   vals_out: torch.Tensor | None = None, begin_bit: int = 0, end_bit: int | None = None,
                   descending: bool = False, temp: torch.Tensor | None = None, key_type: int | None = None,
                   stream=None, return_temp: bool = False):
    """Stable LSD radix sort of (key, value) pairs with 4- or 8-byte values; returns (keys_out, vals_out)."""
    kind = _kind(keys_in, key_type)
    n = keys_in.numel()
    _check_tensor(keys_in, n, "keys_in")
    _check_tensor(vals_in, n, "vals_in")
    if vals_in.element_size() not in (4, 8):
        raise ValueError("values must be 4- or 8-byte elements")
    if keys_out is None:
        keys_out = torch.empty_like(keys_in)
    if vals_out is None:
        vals_out = torch.empty_like(vals_in)
    _check_tensor(keys_out, n, "keys_out")
    _check_tensor(vals_out, n, "vals_out")
    if end_bit is None:
        end_bit = 8 * _KIND_BYTES[kind]
    args = (kind, _ptr(keys_in), _ptr(keys_out), _ptr(vals_in), _ptr(vals_out), n, begin_bit, end_bit,
            int(bool(descending)), _stream(stream))
    fn = load().gbs_sort_pairs64 if vals_in.element_size() == 8 else load().gbs_sort_pairs
    temp = _run(fn, args, temp, "gbs_sort_pairs")
    return (keys_out, vals_out, temp) if return_temp else (keys_out, vals_out)


def gbs_segmented_sort(keys_in: torch.Tensor, num_segments: int, segment_len: int,
                       keys_out: torch.Tensor | None = None, descending: bool = False,
                       temp: torch.Tensor | None = None, key_type: int | None = None, stream=None,
                       return_temp: bool = False):
    """Sort each of num_segments consecutive segments of segment_len keys (bitonic network up to
    GBS_MAX_SEGMENT_LEN keys per segment, the radix sort segment by segment above)."""
    kind = _kind(keys_in, key_type)
    n = num_segments * segment_len
    _check_tensor(keys_in, n, "keys_in")
    if keys_out is None:
        keys_out = torch.empty_like(keys_in)
    _check_tensor(keys_out, n, "keys_out")
    args = (kind, _ptr(keys_in), _ptr(keys_out), num_segments, segment_len, int(bool(descending)), _stream(stream))
    temp = _run(load().gbs_segmented_sort, args, temp, "gbs_segmented_sort")
    return (keys_out, temp) if return_temp else keys_out


def gbs_segmented_sort_offsets(keys_in: torch.Tensor, offsets, keys_out: torch.Tensor | None = None,
                               descending: bool = False, temp: torch.Tensor | None = None,
                               key_type: int | None = None, stream=None, return_temp: bool = False):
    """Sorts each segment [offsets[s], offsets[s+1]) of keys_in independently (any lengths).

    offsets: host sequence of num_segments + 1 non-decreasing integers (list, numpy or CPU tensor).
    keys_out may be keys_in; None allocates a copy of keys_in, so keys outside the segments keep
    their values."""
    kind = _kind(keys_in, key_type)
    n = keys_in.numel()
    _check_tensor(keys_in, n, "keys_in")
    if isinstance(offsets, torch.Tensor):
        offsets = offsets.cpu().numpy()
    offs = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64)).astype(np.uint64)
    if offs.ndim != 1 or offs.size < 1:
        raise ValueError("offsets must hold num_segments + 1 entries")
    if offs.size > 1 and int(offs[-1]) > n:
        raise ValueError("offsets reach past the end of keys_in")
    if keys_out is None:
        keys_out = keys_in.clone()
    _check_tensor(keys_out, n, "keys_out")
    args = (kind, _ptr(keys_in), _ptr(keys_out), offs.size - 1, ctypes.c_void_p(offs.ctypes.data),
            int(bool(descending)), _stream(stream))
    temp = _run(load().gbs_segmented_sort_offsets, args, temp, "gbs_segmented_sort_offsets")
    return (keys_out, temp) if return_temp else keys_out


def gbs_digit_histograms(keys: torch.Tensor, begin_bit: int = 0, end_bit: int | None = None,
                         descending: bool = False, temp: torch.Tensor | None = None,
                         key_type: int | None = None, stream=None) -> torch.Tensor:
    """[passes, 256] uint32 digit counts computed by the upfront-histogram kernel."""
    kind = _kind(keys, key_type)
    n = keys.numel()
    _check_tensor(keys, n, "keys")
    if end_bit is None:
        end_bit = 8 * _KIND_BYTES[kind]
    passes = (end_bit - begin_bit + 7) // 8
    hist = torch.zeros((max(passes, 1), 256), dtype=torch.int32, device="cuda")
    args = (kind, _ptr(keys), n, begin_bit, end_bit, int(bool(descending)), _ptr(hist), _stream(stream))
    _run(load().gbs_digit_histograms, args, temp, "gbs_digit_histograms")
    return hist[:passes]


def gbs_sort_keys_noalloc(keys_in: torch.Tensor, keys_out: torch.Tensor, begin_bit: int = 0,
                          end_bit: int | None = None, descending: bool = False, key_type: int | None = None,
                          stream=None) -> torch.Tensor:
    """gbs_sort_keys without a work buffer, for callers that cannot allocate device memory.

    keys_out must be allocated by the caller (it may be keys_in); nothing is
    allocated here either.  n <= GBS_NOALLOC_MAX_KEYS; calls share one
    library-owned scratch array, so they must not overlap on the GPU."""
    kind = _kind(keys_in, key_type)
    n = keys_in.numel()
    _check_tensor(keys_in, n, "keys_in")
    _check_tensor(keys_out, n, "keys_out")
    if end_bit is None:
        end_bit = 8 * _KIND_BYTES[kind]
    st = load().gbs_sort_keys_noalloc(kind, _ptr(keys_in), _ptr(keys_out), n, begin_bit, end_bit,
                                      int(bool(descending)), _stream(stream))
    if st != GBS_OK:
        raise GbsError(st, "gbs_sort_keys_noalloc")
    return keys_out


def gbs_get_status_noalloc(stream=None) -> int:
    """Synchronises the stream; GBS_ERR_TIMEOUT if the last gbs_sort_keys_noalloc call on the
    current device timed out."""
    return load().gbs_get_status_noalloc(_stream(stream))


def gbs_get_status(temp: torch.Tensor, stream=None) -> int:
    """Synchronises the stream; GBS_ERR_TIMEOUT if the last call on this work buffer timed out."""
    return load().gbs_get_status(_ptr(temp), temp.numel(), _stream(stream))


def gbs_debug_set_lookback_fault(pass_index: int, tile: int, spin_limit: int) -> None:
    load().gbs_debug_set_lookback_fault(pass_index, tile, spin_limit)


def gbs_debug_set_radix_bits(bits: int) -> None:
    """8 (default) or 11: digit width of later keys-only radix sorts below 2^29 keys (test hook)."""
    load().gbs_debug_set_radix_bits(bits)


def gbs_debug_last_launch_count() -> int:
    return load().gbs_debug_last_launch_count()


_timing_keepalive = None


def gbs_debug_set_timing_events(events) -> None:
    """events: list of torch.cuda.Event(enable_timing=True), or None to switch the hook off.

    torch creates an event's CUDA handle on its first record, so unrecorded
    events are recorded once here first."""
    global _timing_keepalive
    if not events:
        _timing_keepalive = None
        load().gbs_debug_set_timing_events(None, 0)
        return
    for e in events:
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _timing_keepalive = (arr, list(events))
    load().gbs_debug_set_timing_events(arr, len(events))


def gbs_debug_radix_tile_keys(key_bytes: int, pairs: bool = False, value_bytes: int | None = None) -> int:
    """Keys per radix tile; value_bytes (0, 4 or 8) overrides pairs (4-byte values)."""
    vb = value_bytes if value_bytes is not None else (4 if pairs else 0)
    return load().gbs_debug_radix_tile_keys(key_bytes, vb)
