"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every symbol the headers declare; argument checks and the work-buffer
size query return the documented status codes without launching anything."""
import ctypes
import os
import re

import pytest

from sorting_lsd_radix_gb300 import build as gbuild
from sorting_lsd_radix_gb300 import gbsort

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gbsort.load()


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(gbs_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert {"gbs_sort_keys", "gbs_sort_pairs", "gbs_segmented_sort", "gbs_get_status"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(gbsort.EXPORTS)


def test_version_and_status_strings(lib):
    assert gbsort.gbs_version() == "0.1.0"
    assert gbsort.status_string(gbsort.GBS_ERR_TEMP_TOO_SMALL) == "GBS_ERR_TEMP_TOO_SMALL"
    assert gbsort.status_string(99) == "GBS_ERR_UNKNOWN"


def _query(lib, fn, *args):
    need = ctypes.c_size_t(0)
    st = getattr(lib, fn)(None, ctypes.byref(need), *args)
    return st, need.value


def test_parity_sizes_straddle_the_launch_shapes_tiles(lib):
    from tests import test_gpu_parity as tp
    assert gbsort.gbs_debug_radix_tile_keys(4) == tp.TILE32
    assert gbsort.gbs_debug_radix_tile_keys(4, value_bytes=4) == tp.TILE32
    assert gbsort.gbs_debug_radix_tile_keys(8) == tp.TILE64
    assert gbsort.gbs_debug_radix_tile_keys(8, value_bytes=4) == tp.TILE64P
    assert gbsort.gbs_debug_radix_tile_keys(4, value_bytes=8) == tp.TILE64P
    assert gbsort.gbs_debug_radix_tile_keys(8, value_bytes=8) == tp.TILE64V64
    for t in (tp.TILE32, tp.TILE64, tp.TILE64P, tp.TILE64V64):
        assert {t - 1, t, t + 1} <= set(tp.SIZES)


def test_temp_query_sizes(lib):
    n = 10**6
    st, need = _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, n, 0, 32, 0, None)
    assert st == gbsort.GBS_OK
    tile = gbsort.gbs_debug_radix_tile_keys(4)
    tiles = (n + tile - 1) // tile
    # header + 2 histogram blocks + status words + one scratch copy of the keys
    assert need >= 256 + 2 * 8 * 256 * 4 + tiles * 1024 + 4 * n
    assert need < 256 + 2 * 8 * 256 * 4 + tiles * 1024 + 4 * n + 4 * 256
    st2, need2 = _query(lib, "gbs_sort_pairs", gbsort.GBS_U64, None, None, None, None, n, 0, 64, 0, None)
    assert st2 == gbsort.GBS_OK and need2 >= 8 * n + 4 * n
    st5, need5 = _query(lib, "gbs_sort_pairs64", gbsort.GBS_U32, None, None, None, None, n, 0, 32, 0, None)
    assert st5 == gbsort.GBS_OK and need5 >= 4 * n + 8 * n
    assert gbsort.gbs_debug_radix_tile_keys(4, value_bytes=8) * 12 <= 64 * 1024  # 64-bit value tile fits
    for kt in (gbsort.GBS_I64, gbsort.GBS_F64):
        st4, need4 = _query(lib, "gbs_sort_keys", kt, None, None, n, 0, 64, 1, None)
        assert st4 == gbsort.GBS_OK and need4 >= 8 * n
        assert _query(lib, "gbs_sort_keys", kt, None, None, n, 0, 65, 0, None)[0] == gbsort.GBS_ERR_INVALID_ARG
    # from 2^29 keys on, the look-back status words are 64-bit: 2 KiB per tile
    for big, per_tile in (((1 << 29) - 1, 1024), (1 << 29, 2048), (gbsort.GBS_MAX_RADIX_KEYS, 2048)):
        st6, need6 = _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, big, 0, 32, 0, None)
        tiles = (big + tile - 1) // tile
        assert st6 == gbsort.GBS_OK
        assert 256 + 2 * 8 * 256 * 4 + tiles * per_tile + 4 * big <= need6
        assert need6 < 256 + 2 * 8 * 256 * 4 + tiles * per_tile + 4 * big + 4 * 256
    st3, need3 = _query(lib, "gbs_segmented_sort", gbsort.GBS_U32, None, None, 16, 1024, 0, None)
    assert st3 == gbsort.GBS_OK and need3 == 256


def test_host_entry_temp_holds_sort_buffer_and_device_keys(lib):
    n = 10**6
    _, sort_need = _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, n, 0, 32, 0, None)
    st, need = _query(lib, "gbs_sort_keys_host", gbsort.GBS_U32, None, None, n, 0, 32, 0, None)
    assert st == gbsort.GBS_OK
    assert sort_need + 4 * n <= need < sort_need + 4 * n + 2 * 256
    st, need64 = _query(lib, "gbs_sort_keys_host", gbsort.GBS_U64, None, None, n, 8, 40, 1, None)
    assert st == gbsort.GBS_OK and need64 >= 2 * 8 * n


def test_host_entry_rejects_bad_arguments(lib):
    assert _query(lib, "gbs_sort_keys_host", 9, None, None, 10, 0, 8, 0, None)[0] == gbsort.GBS_ERR_INVALID_ARG
    assert _query(lib, "gbs_sort_keys_host", gbsort.GBS_I32, None, None, 10, 4, 40, 0, None)[0] == \
        gbsort.GBS_ERR_INVALID_ARG
    assert _query(lib, "gbs_sort_keys_host", gbsort.GBS_U32, None, None, gbsort.GBS_MAX_RADIX_KEYS + 1, 0, 32,
                  0, None)[0] == gbsort.GBS_ERR_UNSUPPORTED
    fake = ctypes.c_void_p(1 << 40)  # never dereferenced: the checks fail first
    have = ctypes.c_size_t(100)
    assert lib.gbs_sort_keys_host(fake, ctypes.byref(have), gbsort.GBS_U32, fake, fake, 1000, 0, 32, 0, None) == \
        gbsort.GBS_ERR_TEMP_TOO_SMALL
    big = ctypes.c_size_t(1 << 30)
    assert lib.gbs_sort_keys_host(fake, ctypes.byref(big), gbsort.GBS_U32, None, fake, 1000, 0, 32, 0, None) == \
        gbsort.GBS_ERR_INVALID_ARG


def _batch_args(sizes, ins=None, outs=None):
    k = max(len(sizes), 1)
    fake = 1 << 40  # never dereferenced: the checks fail first
    ins = (ctypes.c_void_p * k)(*(ins if ins is not None else [fake] * len(sizes)))
    outs = (ctypes.c_void_p * k)(*(outs if outs is not None else [fake] * len(sizes)))
    ns = (ctypes.c_size_t * k)(*sizes)
    return ins, outs, ns


def test_host_batch_temp_holds_one_sort_buffer_and_three_key_buffers(lib):
    sizes = [10**6, 7, 3 * 10**6 + 5, 0]
    ins, outs, ns = _batch_args(sizes)
    _, sort_need = _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, max(sizes), 0, 32, 0, None)
    st, need = _query(lib, "gbs_sort_keys_host_batch", gbsort.GBS_U32, ins, outs, ns, len(sizes), 0, 32, 0, None)
    assert st == gbsort.GBS_OK
    slot = (4 * max(sizes) + 255) // 256 * 256
    assert need - 3 * slot in range(sort_need, sort_need + 256)
    # 64-bit keys: the slots hold 8 bytes per key
    _, sort64 = _query(lib, "gbs_sort_keys", gbsort.GBS_F64, None, None, max(sizes), 0, 64, 1, None)
    st, need64 = _query(lib, "gbs_sort_keys_host_batch", gbsort.GBS_F64, ins, outs, ns, len(sizes), 0, 64, 1, None)
    assert st == gbsort.GBS_OK and need64 - 3 * ((8 * max(sizes) + 255) // 256 * 256) in range(sort64, sort64 + 256)
    # an empty batch needs the header of a sort of no keys
    st, need0 = _query(lib, "gbs_sort_keys_host_batch", gbsort.GBS_U32, None, None, None, 0, 0, 32, 0, None)
    assert st == gbsort.GBS_OK and need0 == _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, 0, 0, 32, 0,
                                                   None)[1]


def test_host_batch_rejects_bad_arguments(lib):
    ins, outs, ns = _batch_args([1000, 2000])
    q = lambda *a: _query(lib, "gbs_sort_keys_host_batch", *a)[0]
    assert q(9, ins, outs, ns, 2, 0, 8, 0, None) == gbsort.GBS_ERR_INVALID_ARG
    assert q(gbsort.GBS_I32, ins, outs, ns, 2, 4, 40, 0, None) == gbsort.GBS_ERR_INVALID_ARG
    assert q(gbsort.GBS_U32, ins, outs, None, 2, 0, 32, 0, None) == gbsort.GBS_ERR_INVALID_ARG
    assert q(gbsort.GBS_U32, None, outs, ns, 2, 0, 32, 0, None) == gbsort.GBS_ERR_INVALID_ARG
    assert q(gbsort.GBS_U32, ins, None, ns, 2, 0, 32, 0, None) == gbsort.GBS_ERR_INVALID_ARG
    big = _batch_args([10, gbsort.GBS_MAX_RADIX_KEYS + 1])
    assert q(gbsort.GBS_U32, *big, 2, 0, 32, 0, None) == gbsort.GBS_ERR_UNSUPPORTED
    fake = ctypes.c_void_p(1 << 40)
    small = ctypes.c_size_t(1000)
    assert lib.gbs_sort_keys_host_batch(fake, ctypes.byref(small), gbsort.GBS_U32, ins, outs, ns, 2, 0, 32, 0,
                                        None) == gbsort.GBS_ERR_TEMP_TOO_SMALL
    roomy = ctypes.c_size_t(1 << 30)
    nul = _batch_args([1000, 2000], ins=[1 << 40, 0])
    assert lib.gbs_sort_keys_host_batch(fake, ctypes.byref(roomy), gbsort.GBS_U32, *nul, 2, 0, 32, 0,
                                        None) == gbsort.GBS_ERR_INVALID_ARG
    unaligned = ctypes.c_void_p((1 << 40) + 8)
    assert lib.gbs_sort_keys_host_batch(unaligned, ctypes.byref(roomy), gbsort.GBS_U32, ins, outs, ns, 2, 0, 32, 0,
                                        None) == gbsort.GBS_ERR_INVALID_ARG


def test_host_batch_binding_checks_its_arguments(lib):
    torch = pytest.importorskip("torch")
    a32, b32 = torch.zeros(3, dtype=torch.int32), torch.zeros(5, dtype=torch.int32)
    with pytest.raises(ValueError):  # one dtype for the whole batch
        gbsort.gbs_sort_keys_host_batch([a32, torch.zeros(3, dtype=torch.int64)])
    with pytest.raises(ValueError):  # one output per input
        gbsort.gbs_sort_keys_host_batch([a32, b32], [torch.zeros(3, dtype=torch.int32)])
    with pytest.raises(ValueError):  # outputs shaped like their inputs
        gbsort.gbs_sort_keys_host_batch([a32, b32], [torch.zeros(3, dtype=torch.int32), torch.zeros(4, dtype=torch.int32)])
    with pytest.raises(ValueError):  # contiguous host tensors only
        gbsort.gbs_sort_keys_host_batch([a32[::2]])


def _offsets(values):
    a = (ctypes.c_uint64 * len(values))(*values)
    return a


def test_segmented_offsets_temp_and_arguments(lib):
    small = _offsets([0, 10, 10, 5000, 21384])  # longest 16384: bitonic only
    st, need_small = _query(lib, "gbs_segmented_sort_offsets", gbsort.GBS_U32, None, None, 4, small, 0, None)
    assert st == gbsort.GBS_OK and need_small < 4096
    big = _offsets([0, 10, 100010, 100011])     # one segment of 10^5 keys: radix work area
    st, need_big = _query(lib, "gbs_segmented_sort_offsets", gbsort.GBS_U32, None, None, 3, big, 0, None)
    _, radix = _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, 100000, 0, 32, 0, None)
    assert st == gbsort.GBS_OK and need_big >= radix
    bad = _offsets([0, 10, 5, 20])
    assert _query(lib, "gbs_segmented_sort_offsets", gbsort.GBS_U32, None, None, 3, bad, 0, None)[0] == \
        gbsort.GBS_ERR_INVALID_ARG
    assert _query(lib, "gbs_segmented_sort_offsets", gbsort.GBS_U32, None, None, 3, None, 0, None)[0] == \
        gbsort.GBS_ERR_INVALID_ARG
    huge = _offsets([0, gbsort.GBS_MAX_RADIX_KEYS + 1])
    assert _query(lib, "gbs_segmented_sort_offsets", gbsort.GBS_U64, None, None, 1, huge, 0, None)[0] == \
        gbsort.GBS_ERR_UNSUPPORTED
    st, need0 = _query(lib, "gbs_segmented_sort_offsets", gbsort.GBS_F64, None, None, 0, None, 0, None)
    assert st == gbsort.GBS_OK and need0 > 0


@pytest.mark.parametrize("begin,end", [(-1, 8), (9, 8), (0, 33)])
def test_bad_bit_range(lib, begin, end):
    st, _ = _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, 10, begin, end, 0, None)
    assert st == gbsort.GBS_ERR_INVALID_ARG


def test_bad_key_type_and_limits(lib):
    assert _query(lib, "gbs_sort_keys", 7, None, None, 10, 0, 8, 0, None)[0] == gbsort.GBS_ERR_INVALID_ARG
    assert _query(lib, "gbs_sort_keys", 6, None, None, 10, 0, 8, 0, None)[0] == gbsort.GBS_ERR_INVALID_ARG
    assert _query(lib, "gbs_sort_keys", gbsort.GBS_U32, None, None, gbsort.GBS_MAX_RADIX_KEYS + 1, 0, 32, 0,
                  None)[0] == gbsort.GBS_ERR_UNSUPPORTED
    # segments longer than one CTA's network take the radix path: a larger work buffer
    st_small, need_small = _query(lib, "gbs_segmented_sort", gbsort.GBS_U32, None, None, 4, 16384, 0, None)
    st_long, need_long = _query(lib, "gbs_segmented_sort", gbsort.GBS_U32, None, None, 4, 16385, 0, None)
    assert st_small == st_long == gbsort.GBS_OK and need_long > need_small + 4 * 16385
    assert _query(lib, "gbs_segmented_sort", gbsort.GBS_U32, None, None, 1, gbsort.GBS_MAX_RADIX_KEYS + 1, 0,
                  None)[0] == gbsort.GBS_ERR_UNSUPPORTED
    assert lib.gbs_sort_keys(None, None, gbsort.GBS_U32, None, None, 10, 0, 32, 0, None) == \
        gbsort.GBS_ERR_INVALID_ARG


def test_temp_too_small_and_misaligned(lib):
    fake = ctypes.c_void_p(1 << 40)  # never dereferenced: the checks fail first
    have = ctypes.c_size_t(100)
    assert lib.gbs_sort_keys(fake, ctypes.byref(have), gbsort.GBS_U32, fake, fake, 1000, 0, 32, 0, None) == \
        gbsort.GBS_ERR_TEMP_TOO_SMALL
    big = ctypes.c_size_t(1 << 30)
    odd = ctypes.c_void_p((1 << 40) + 16)
    assert lib.gbs_sort_keys(odd, ctypes.byref(big), gbsort.GBS_U32, fake, fake, 1000, 0, 32, 0, None) == \
        gbsort.GBS_ERR_INVALID_ARG


def test_oracle_and_library_share_nothing():
    # the oracle and the CUDA sources never include or import each other
    csrc = os.path.join(ROOT, "sorting_lsd_radix_gb300", "csrc")
    for f in os.listdir(csrc):
        assert "oracle" not in open(os.path.join(csrc, f)).read().lower(), f
    for f in ("oracle.c", "oracle.h", "__init__.py"):
        text = open(os.path.join(ROOT, "oracle", f)).read()
        assert "gbsort" not in text and "sorting_lsd_radix_gb300" not in text and "csrc" not in text, f
    for f in ("gbsort.py", "build.py", "__init__.py"):
        text = open(os.path.join(ROOT, "sorting_lsd_radix_gb300", f)).read()
        assert "import oracle" not in text and "from oracle" not in text, f
