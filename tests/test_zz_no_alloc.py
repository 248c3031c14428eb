"""The allocation-free sort entry point.

gbs_sort_keys_noalloc serves callers that cannot allocate device memory (its
scratch is a fixed array inside the library).  Its output must equal the
oracle's stable sort and what gbs_sort_keys returns, on consecutive calls
that reuse that array; in-place calls with an odd number of digit passes
(which end in the scratch array and need the final copy), the early returns
for n <= 1 and empty bit ranges, the size limit and the timeout report of
gbs_get_status_noalloc are checked too.  This file runs last so that a
failure here does not hide the other tests' results."""
import ctypes

import numpy as np
import pytest

import oracle
from sorting_lsd_radix_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sorting_lsd_radix_gb300 import build as gbuild
    gbuild.build()
    from sorting_lsd_radix_gb300 import gbsort
    gbsort.load()
    yield gbsort
    gbsort.gbs_debug_set_lookback_fault(-1, 0, 0)


def _u(a):
    return a.view(np.uint64 if a.dtype.itemsize == 8 else np.uint32)


def _keys(kind, n, seed):
    if kind == "u32":
        return wl.low_entropy_u32(n, seed)
    if kind == "f32":
        return wl.normal_mix_f32(n, seed)
    if kind == "u64":
        return wl.priority_u64(n, seed)
    return wl.uniform_i32(n, seed)


@pytest.mark.parametrize("case", [
    ("u32", 300001, 0, 32, False),
    ("f32", 1 << 20, 0, 32, True),
    ("u64", 200003, 0, 52, False),
    ("i32", 77777, 4, 28, True),
])
def test_noalloc_matches_oracle_and_regular_sort_twice(g, case):
    kind, n, b, e, desc = case
    for call, seed in enumerate([wl.seed_for(50, 1), wl.seed_for(50, 2)]):  # two calls share the array
        keys = _keys(kind, n, seed)
        d = torch.from_numpy(keys).cuda()
        out = torch.empty_like(d)
        g.gbs_sort_keys_noalloc(d, out, begin_bit=b, end_bit=e, descending=desc)
        assert g.gbs_get_status_noalloc() == g.GBS_OK
        got = _u(out.cpu().numpy())
        assert np.array_equal(got, _u(oracle.sort_keys(keys, b, e, descending=desc))), (kind, call)
        regular = g.gbs_sort_keys(d, begin_bit=b, end_bit=e, descending=desc)
        assert np.array_equal(got, _u(regular.cpu().numpy())), (kind, call)


@pytest.mark.parametrize("case", [
    ("u32", 100000, 0, 32),  # four passes: the last one lands in the caller's array
    ("i32", 99999, 4, 28),   # three passes: ends in the scratch array, then the final copy
    ("u64", 50001, 8, 48),   # five passes
])
def test_noalloc_in_place(g, case):
    kind, n, b, e = case
    keys = _keys(kind, n, wl.seed_for(50, 3))
    d = torch.from_numpy(keys).cuda()
    g.gbs_sort_keys_noalloc(d, d, begin_bit=b, end_bit=e)
    assert g.gbs_get_status_noalloc() == g.GBS_OK
    assert np.array_equal(_u(d.cpu().numpy()), _u(oracle.sort_keys(keys, b, e)))


def test_noalloc_trivial_calls(g):
    keys = wl.uniform_u32(1000, wl.seed_for(50, 4))
    d = torch.from_numpy(keys).cuda()
    for n in (0, 1):  # nothing to sort: a copy of n keys at most
        out = torch.full((n,), 7, dtype=torch.uint32, device="cuda")
        g.gbs_sort_keys_noalloc(d[:n], out)
        assert np.array_equal(out.cpu().numpy(), keys[:n])
    out = torch.empty_like(d)
    g.gbs_sort_keys_noalloc(d, out, begin_bit=9, end_bit=9)  # empty bit range: a copy
    assert np.array_equal(out.cpu().numpy(), keys)
    assert g.gbs_get_status_noalloc() == g.GBS_OK


def test_noalloc_limit_and_timeout_report(g):
    lib = g.load()
    big = g.GBS_NOALLOC_MAX_KEYS + 1
    # rejected before anything is launched: the pointers are never touched
    st = lib.gbs_sort_keys_noalloc(g.GBS_U32, ctypes.c_void_p(1 << 40), ctypes.c_void_p(1 << 40), big, 0, 32, 0,
                                   None)
    assert st == g.GBS_ERR_UNSUPPORTED
    # a tile that never publishes its look-back status: the bounded wait gives up, the header
    # records the timeout, the status query reports it, and the next call is correct again
    n = 6 * g.gbs_debug_radix_tile_keys(4) + 5
    keys = wl.uniform_u32(n, wl.seed_for(50, 5))
    d = torch.from_numpy(keys).cuda()
    out = torch.empty_like(d)
    g.gbs_debug_set_lookback_fault(1, 2, 1 << 12)
    try:
        g.gbs_sort_keys_noalloc(d, out, begin_bit=0, end_bit=24)
        assert g.gbs_get_status_noalloc() == g.GBS_ERR_TIMEOUT
    finally:
        g.gbs_debug_set_lookback_fault(-1, 0, 0)
    g.gbs_sort_keys_noalloc(d, out, begin_bit=0, end_bit=24)
    assert g.gbs_get_status_noalloc() == g.GBS_OK
    assert np.array_equal(out.cpu().numpy(), oracle.sort_keys(keys, 0, 24))
