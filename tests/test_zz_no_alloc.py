"""The allocation-free sort entry point against the regular one.

gbs_sort_keys_noalloc serves callers that cannot allocate device memory (its
scratch is a fixed array inside the library).  It must return exactly what
gbs_sort_keys returns, on consecutive calls that reuse that array, and refuse
sizes beyond its maximum.  This file runs last so that a failure here does
not hide the other tests' results."""
import ctypes

import numpy as np
import pytest

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
    return gbsort


def _u(a):
    return a.view(np.uint64 if a.dtype.itemsize == 8 else np.uint32)


@pytest.mark.parametrize("case", [
    ("u32", 300001, 0, 32, False),
    ("f32", 1 << 20, 0, 32, True),
    ("u64", 200003, 0, 52, False),
    ("i32", 77777, 4, 28, True),
])
def test_noalloc_matches_regular_sort_twice(g, case):
    kind, n, b, e, desc = case
    seeds = [wl.seed_for(50, 1), wl.seed_for(50, 2)]
    for call, seed in enumerate(seeds):  # two calls in a row share the library's scratch array
        if kind == "u32":
            keys = wl.low_entropy_u32(n, seed)
        elif kind == "f32":
            keys = wl.normal_mix_f32(n, seed)
        elif kind == "u64":
            keys = wl.priority_u64(n, seed)
        else:
            keys = wl.uniform_i32(n, seed)
        d = torch.from_numpy(keys).cuda()
        want = g.gbs_sort_keys(d, begin_bit=b, end_bit=e, descending=desc)
        out = torch.empty_like(d)
        g.gbs_sort_keys_noalloc(d, out, begin_bit=b, end_bit=e, descending=desc)
        torch.cuda.synchronize()
        assert np.array_equal(_u(out.cpu().numpy()), _u(want.cpu().numpy())), (kind, call)


def test_noalloc_in_place_and_limits(g):
    keys = wl.uniform_u32(100000, wl.seed_for(50, 3))
    d = torch.from_numpy(keys).cuda()
    want = g.gbs_sort_keys(d.clone())
    g.gbs_sort_keys_noalloc(d, d)
    assert np.array_equal(d.cpu().numpy(), want.cpu().numpy())
    lib = g.load()
    big = g.GBS_NOALLOC_MAX_KEYS + 1
    # rejected before anything is launched: the pointers are never touched
    st = lib.gbs_sort_keys_noalloc(g.GBS_U32, ctypes.c_void_p(1 << 40), ctypes.c_void_p(1 << 40), big, 0, 32, 0,
                                   None)
    assert st == g.GBS_ERR_UNSUPPORTED
