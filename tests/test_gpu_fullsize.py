"""GPU parity at the full sizes of the benchmark workloads.

Each configuration is sorted by the CUDA library with the same launch shapes the
benchmark uses, and compared bit for bit with the oracle on the same seeded
input (the whole output where the oracle finishes in seconds; for the
4096 x 16384 segmented case, every segment is checked for order and content and
a sample of segments is compared with the oracle's bitonic network)."""
import numpy as np
import pytest

import oracle
from sorting_lsd_radix_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]


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


def _sorted_u32(g, keys, **kw):
    d = torch.from_numpy(keys).cuda()
    out, temp = g.gbs_sort_keys(d, return_temp=True, **kw)
    assert g.gbs_get_status(temp) == g.GBS_OK
    res = out.cpu().numpy()
    del d, out, temp
    torch.cuda.empty_cache()
    return res


def test_config1_u32_2p20_uniform(g):
    keys = wl.uniform_u32(1 << 20, wl.seed_for(1, 0))
    assert np.array_equal(_sorted_u32(g, keys), oracle.sort_keys(keys))


@pytest.mark.parametrize("desc", [False, True])
def test_config2_segmented_16384x1024(g, desc):
    segs, L = 16384, 1024
    keys = wl.uniform_u32(segs * L, wl.seed_for(2, 0))
    out = g.gbs_segmented_sort(torch.from_numpy(keys).cuda(), segs, L, descending=desc).cpu().numpy()
    assert np.array_equal(out, oracle.segmented_sort(keys, segs, L, descending=desc))


@pytest.mark.parametrize("desc", [False, True])
def test_config2_segmented_4096x16384(g, desc):
    segs, L = 4096, 16384
    keys = wl.uniform_u32(segs * L, wl.seed_for(2, 1))
    out = g.gbs_segmented_sort(torch.from_numpy(keys).cuda(), segs, L, descending=desc).cpu().numpy()
    rows_in = keys.reshape(segs, L)
    rows_out = out.reshape(segs, L)
    # every segment: ordered, and the same multiset as its input
    d = np.diff(rows_out.astype(np.int64), axis=1)
    assert (d <= 0).all() if desc else (d >= 0).all()
    assert np.array_equal(np.sort(rows_out, axis=1), np.sort(rows_in, axis=1))
    # sampled segments: exactly the oracle's network output
    pick = (wl.uniform_u32(64, wl.seed_for(2, 2)) % np.uint32(segs)).astype(np.int64)
    for s in pick:
        assert np.array_equal(rows_out[s], oracle.bitonic_sort(rows_in[s], descending=desc))


N3 = 100_000_000


@pytest.mark.parametrize("dist", list(wl.DISTRIBUTIONS_U32))
def test_config3_u32_1e8(g, dist):
    keys = wl.DISTRIBUTIONS_U32[dist](N3, wl.seed_for(3, 1))
    assert np.array_equal(_sorted_u32(g, keys), oracle.sort_keys(keys)), dist


def test_config3_u32_1e8_low16(g):
    keys = wl.uniform_u32(N3, wl.seed_for(3, 0))
    assert np.array_equal(_sorted_u32(g, keys, begin_bit=0, end_bit=16), oracle.sort_keys(keys, 0, 16))


def test_config4_pairs_u64_2p27_stable(g):
    n = 1 << 27
    keys = wl.priority_u64(n, wl.seed_for(4, 0))
    vals = np.arange(n, dtype=np.uint32)
    ko, vo, temp = g.gbs_sort_pairs(torch.from_numpy(keys).cuda(), torch.from_numpy(vals).cuda(), return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK
    ko, vo = ko.cpu().numpy(), vo.cpu().numpy()
    ek, ev = oracle.sort_pairs(keys, vals)
    assert np.array_equal(ko, ek)
    assert np.array_equal(vo, ev)
    # stability by definition: within equal keys the original indices increase
    same = ko[1:] == ko[:-1]
    assert (vo[1:][same] > vo[:-1][same]).all()


@pytest.mark.parametrize("kind", ["f32", "i32"])
@pytest.mark.parametrize("desc", [False, True])
def test_config5_2p28(g, kind, desc):
    n = 1 << 28
    keys = wl.normal_mix_f32(n, wl.seed_for(5, 0)) if kind == "f32" else wl.uniform_i32(n, wl.seed_for(5, 1))
    d = torch.from_numpy(keys).cuda()
    out, temp = g.gbs_sort_keys(d, descending=desc, return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK
    got = out.cpu().numpy()
    del d, out, temp
    torch.cuda.empty_cache()
    assert np.array_equal(_u(got), _u(oracle.sort_keys(keys, descending=desc)))


@pytest.mark.parametrize("dist", ["uniform", "all_equal"])
def test_largest_narrow_status_size_u32(g, dist):
    # 2^29 - 1 keys, the largest sort whose look-back status words are 32-bit: their 29-bit
    # counts reach the limit (all-equal keys put every key in one digit; uniform keys make the
    # largest prefixes near n)
    n = (1 << 29) - 1
    keys = wl.uniform_u32(n, wl.seed_for(3, 7)) if dist == "uniform" else wl.all_equal_u32(n, wl.seed_for(3, 8))
    got = _sorted_u32(g, keys)
    assert np.array_equal(got, oracle.sort_keys(keys))


@pytest.mark.parametrize("dist", ["uniform", "all_equal", "and4"])
def test_wide_status_2p30_plus_7_u32(g, dist):
    # 2^30 + 7 keys take the 64-bit status words.  "and4": the AND of four uniform draws, so
    # digit value 0 holds about 60% of the keys in every pass and the inclusive prefixes of
    # that digit pass 2^29 while every pass stays active
    n = (1 << 30) + 7
    if dist == "uniform":
        keys = wl.uniform_u32(n, wl.seed_for(3, 9))
    elif dist == "all_equal":
        keys = wl.all_equal_u32(n, wl.seed_for(3, 10))
    else:
        keys = wl.low_entropy_u32(n, wl.seed_for(3, 11))
        keys &= wl.uniform_u32(n, wl.seed_for(3, 12))
    got = _sorted_u32(g, keys)
    want = oracle.sort_keys(keys)
    if dist == "and4":
        assert ((want & np.uint32(0xFF)) == 0).sum() > (1 << 29)  # digit 0 of pass 0 passes 2^29 keys
    assert np.array_equal(got, want)


def _as_signed_order(x):
    """int32 tensor of uint32 bit patterns -> int32 values in the same order as the unsigned keys."""
    return x ^ torch.tensor(-(1 << 31), dtype=torch.int32, device=x.device)


def test_largest_radix_size_u32(g):
    """The largest radix sort the library accepts: 2^32 - 1 u32 keys (16 GiB, 524,288 tiles,
    64-bit status words), drawn on the device (the same SplitMix64 stream as the host generator).
    The oracle cannot sort 2^32 keys in test time, so the result is checked by properties that hold
    at any size, with torch operations only: the output is non-decreasing; each of its four byte
    positions has the input's value counts; and at sampled positions i the output value v satisfies
    #(keys < v) <= i < #(keys <= v), which makes v the i-th smallest key."""
    n = g.GBS_MAX_RADIX_KEYS
    keys = wl.uniform_u32_torch(n, wl.seed_for(3, 13), "cuda")
    # the device draws are the host stream's (checked on a slice)
    assert np.array_equal(keys[:4096].cpu().numpy().view(np.uint32), wl.uniform_u32(4096, wl.seed_for(3, 13)))
    out, temp = g.gbs_sort_keys(keys, return_temp=True, key_type=g.GBS_U32)
    assert g.gbs_get_status(temp) == g.GBS_OK
    del temp
    torch.cuda.empty_cache()
    chunk = 1 << 28
    for start in range(0, n - 1, chunk):
        a = _as_signed_order(out[start:min(n, start + chunk + 1)])
        assert bool((a[1:] >= a[:-1]).all()), start
    for p in range(4):
        hi, ho = torch.zeros(256, dtype=torch.int64, device="cuda"), torch.zeros(256, dtype=torch.int64, device="cuda")
        for start in range(0, n, chunk):
            stop = min(n, start + chunk)
            hi += torch.bincount(((keys[start:stop] >> (8 * p)) & 0xFF).to(torch.int64), minlength=256)
            ho += torch.bincount(((out[start:stop] >> (8 * p)) & 0xFF).to(torch.int64), minlength=256)
        assert torch.equal(hi, ho), p
    rng = np.random.default_rng(wl.seed_for(3, 14))
    for i in [0, n - 1] + [int(x) for x in rng.integers(0, n, 6)]:
        v = _as_signed_order(out[i:i + 1])
        below = at_most = 0
        for start in range(0, n, chunk):
            k = _as_signed_order(keys[start:min(n, start + chunk)])
            below += int((k < v).sum())
            at_most += int((k <= v).sum())
        assert below <= i < at_most, i

