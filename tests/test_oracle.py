"""Pins the CPU oracle to facts fixed outside itself: the pages' worked examples and
printed bit patterns, the 0-1 principle, the network-size closed forms, library
sorts (numpy stable argsort, Python's sorted) and brute force on tiny inputs."""
import itertools
import math

import numpy as np
import pytest

import oracle
from sorting_lsd_radix_gb300 import workloads as wl
from tests import golden_io

KINDS = [np.uint32, np.int32, np.float32, np.uint64, np.int64, np.float64]


# --------------------------------------------------------------------------
# Bitonic network
# --------------------------------------------------------------------------

def test_worked_example():
    rows = dict(golden_io.read("bitonic_worked_example.txt"))
    src = np.array(golden_io.ints(rows["input"]), dtype=np.uint32)
    want = golden_io.ints(rows["ascending"])
    assert oracle.bitonic_sort(src).tolist() == want
    assert oracle.bitonic_sort(src, descending=True).tolist() == want[::-1]
    assert oracle.segmented_sort(src, 1, 8).tolist() == want


def _is_bitonic(seq):
    # rises then falls for some cyclic shift: at most two direction changes around the cycle
    n = len(seq)
    changes = 0
    signs = []
    for i in range(n):
        d = seq[(i + 1) % n] - seq[i]
        if d != 0:
            signs.append(1 if d > 0 else -1)
    for i in range(len(signs)):
        if signs[i] != signs[(i + 1) % len(signs)]:
            changes += 1
    return changes <= 2


def test_page_sequences_are_bitonic_and_merge_sorts_them():
    rows = golden_io.read("bitonic_sequences.txt")
    seqs = [golden_io.ints(v) for k, v in rows if k == "bitonic"]
    for s in seqs:
        assert _is_bitonic(s), s
    for k, v in rows:
        if k == "page_misprint_not_bitonic":
            assert not _is_bitonic(golden_io.ints(v))
    for s in seqs:
        if len(s) & (len(s) - 1) == 0:
            assert oracle.bitonic_merge(np.array(s)).tolist() == sorted(s)
            assert oracle.bitonic_merge(np.array(s), up=False).tolist() == sorted(s, reverse=True)
    assert not _is_bitonic([1, 3, 2, 4])


@pytest.mark.parametrize("cnt", [2, 4, 8, 16, 64, 256])
def test_half_cleaner_property(cnt):
    # bitonic split: first half <= second half, both halves bitonic ("并行排序", §3.2)
    rng = np.random.default_rng(cnt)
    for trial in range(200):
        k = int(rng.integers(0, cnt + 1))
        vals = rng.integers(0, 20, cnt)
        seq = np.concatenate([np.sort(vals[:k]), np.sort(vals[k:])[::-1]])
        seq = np.roll(seq, int(rng.integers(0, cnt)))
        assert _is_bitonic(seq.tolist())
        out = oracle.bitonic_split(seq)
        lo, hi = out[: cnt // 2], out[cnt // 2:]
        assert lo.max() <= hi.min()
        assert _is_bitonic(lo.tolist()) and _is_bitonic(hi.tolist())
        down = oracle.bitonic_split(seq, up=False)
        assert down[: cnt // 2].min() >= down[cnt // 2:].max()


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8, 12, 16])
def test_zero_one_principle_exhaustive(bits):
    # every 0-1 input of length 2^q = bits is sorted ("并行排序", §1.2)
    pats = wl.zero_one_patterns(bits)
    out = oracle.segmented_sort(pats.reshape(-1), pats.shape[0], bits).reshape(pats.shape)
    ones = pats.sum(axis=1)
    want = (np.arange(bits)[None, :] >= (bits - ones)[:, None]).astype(np.uint32)
    assert np.array_equal(out, want)
    outd = oracle.segmented_sort(pats.reshape(-1), pats.shape[0], bits, descending=True).reshape(pats.shape)
    assert np.array_equal(outd, want[:, ::-1])


@pytest.mark.parametrize("p", range(0, 17))
def test_network_size_closed_forms(p):
    n = 1 << p
    keys = wl.uniform_u32(n, wl.seed_for(90, p))
    out, comps, depth = oracle.bitonic_sort(keys, count=True)
    assert comps == n * p * (p + 1) // 4
    assert depth == p * (p + 1) // 2
    assert np.array_equal(out, np.sort(keys))


def test_network_size_page_numbers():
    g = dict(golden_io.read("network_size.txt"))
    p = int(g["p"])
    keys = wl.uniform_u32(1 << p, wl.seed_for(91))
    out, comps, depth = oracle.bitonic_sort(keys, count=True)
    assert depth == int(g["depth"])
    assert comps == int(g["comparators_exact"])
    assert abs(comps - int(g["comparators_approx"])) / comps < 0.01
    assert np.array_equal(out, np.sort(keys))


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 6, 7, 8])
def test_bitonic_all_permutations(n):
    if n == 0:
        assert oracle.bitonic_sort(np.zeros(0, np.uint32)).size == 0
        return
    perms = np.array(list(itertools.permutations(range(n))), dtype=np.uint32).reshape(-1, n)
    out = oracle.segmented_sort(perms.reshape(-1), perms.shape[0], n).reshape(perms.shape)
    assert (out == np.arange(n, dtype=np.uint32)[None, :]).all()
    outd = oracle.segmented_sort(perms.reshape(-1), perms.shape[0], n, descending=True).reshape(perms.shape)
    assert (outd == np.arange(n, dtype=np.uint32)[None, ::-1]).all()


@pytest.mark.parametrize("dtype", KINDS)
@pytest.mark.parametrize("seg_len", [1, 3, 17, 100, 1024])
def test_segmented_matches_library_sort(dtype, seg_len):
    segs = 7
    keys = _sample(dtype, segs * seg_len, 5 + seg_len)
    want = np.stack([_library_sorted_keys(keys[s * seg_len:(s + 1) * seg_len], False) for s in range(segs)])
    got = oracle.segmented_sort(keys, segs, seg_len)
    assert np.array_equal(got.view(_uint_view(dtype)), want.reshape(-1).view(_uint_view(dtype)))
    wantd = np.stack([_library_sorted_keys(keys[s * seg_len:(s + 1) * seg_len], True) for s in range(segs)])
    gotd = oracle.segmented_sort(keys, segs, seg_len, descending=True)
    assert np.array_equal(gotd.view(_uint_view(dtype)), wantd.reshape(-1).view(_uint_view(dtype)))


# --------------------------------------------------------------------------
# Key encodings
# --------------------------------------------------------------------------

def test_page_bit_patterns():
    g = golden_io.read("key_encodings.txt")
    vals = {k: int(v, 0) for k, v in g}
    neg, pos = vals["f32_bits -1.0"], vals["f32_bits 1.0"]
    assert np.array([-1.0, 1.0], np.float32).view(np.uint32).tolist() == [neg, pos]
    assert pos < neg  # raw unsigned order is wrong, as the page says
    assert oracle.transform(oracle.KIND_F32, neg) < oracle.transform(oracle.KIND_F32, pos)
    assert oracle.transform(oracle.KIND_I32, np.uint32(np.int32(-2**31).view(np.uint32))) == vals["i32_code -2147483648"]
    assert oracle.transform(oracle.KIND_I32, 2**31 - 1) == vals["i32_code 2147483647"]


def test_f32_code_order_is_value_order_exhaustive_sample():
    # Every non-NaN float in increasing value order must get strictly increasing codes,
    # with -0.0 just before +0.0.  Walk the floats by value from -inf to +inf.
    neg_bits = np.arange(0xFF800000, 0x7FFFFFFF, -4099, dtype=np.int64)  # -inf .. -0 (descending bits)
    neg_bits = np.append(neg_bits, 0x80000000)
    pos_bits = np.arange(0, 0x7F800001, 4099, dtype=np.int64)
    pos_bits = np.append(pos_bits, 0x7F800000)
    walk = np.concatenate([neg_bits[neg_bits >= 0x80000000], pos_bits]).astype(np.uint32)
    f = walk.view(np.float32)
    assert not np.isnan(f).any()
    assert (np.diff(f.astype(np.float64)) >= 0).all()
    codes = oracle.transform_array(f)
    assert (np.diff(codes.astype(np.int64)) > 0).all()
    assert codes[0] == 0x007FFFFF and codes[-1] == 0xFF800000  # -inf and +inf are the extremes
    z = oracle.transform_array(np.array([-0.0, 0.0], np.float32))
    assert z[0] + 1 == z[1]
    dcodes = oracle.transform_array(f, descending=True)
    assert (np.diff(dcodes.astype(np.int64)) < 0).all()


def test_f64_code_order_is_value_order_sample():
    # Non-NaN doubles in increasing value order (a strided walk over the bit patterns from -inf to
    # +inf, plus the neighbours of every power-of-two boundary near 1.0) get strictly increasing codes.
    step = 0x00005A5A5A5A5A5B  # about 93 thousand doubles of each sign
    neg = np.arange(0xFFF0000000000000, 0x8000000000000000, -step, dtype=np.uint64)
    neg = np.append(neg[neg >= np.uint64(0x8000000000000000)], np.uint64(0x8000000000000000))
    pos = np.append(np.arange(0, 0x7FF0000000000000, step, dtype=np.uint64), np.uint64(0x7FF0000000000000))
    walk = np.concatenate([neg, pos])
    f = walk.view(np.float64)
    assert not np.isnan(f).any()
    assert (np.diff(f) >= 0).all()
    codes = oracle.transform_array(f)
    assert (codes[1:] > codes[:-1]).all()
    assert codes[0] == 0x000FFFFFFFFFFFFF and codes[-1] == 0xFFF0000000000000  # -inf, +inf extremes
    z = oracle.transform_array(np.array([-0.0, 0.0], np.float64))
    assert z[0] + np.uint64(1) == z[1]
    # IEEE-754 patterns of -1.0 and 1.0: raw unsigned order is reversed, code order is not
    neg1, pos1 = np.array([-1.0, 1.0], np.float64).view(np.uint64)
    assert (int(neg1), int(pos1)) == (0xBFF0000000000000, 0x3FF0000000000000)
    assert oracle.transform(oracle.KIND_F64, int(neg1)) < oracle.transform(oracle.KIND_F64, int(pos1))
    dcodes = oracle.transform_array(f, descending=True)
    assert (dcodes[1:] < dcodes[:-1]).all()


def test_i64_code_is_offset_binary():
    ext = np.array([-2**63, -1, 0, 1, 2**63 - 1], dtype=np.int64)
    codes = oracle.transform_array(ext)
    assert codes.tolist() == [0, 2**63 - 1, 2**63, 2**63 + 1, 2**64 - 1]


@pytest.mark.parametrize("dtype", [np.int32, np.float32, np.uint32, np.uint64, np.int64, np.float64])
def test_code_order_matches_native_comparison(dtype):
    a = _sample(dtype, 20000, 11)
    b = _sample(dtype, 20000, 12)
    ca, cb = oracle.transform_array(a), oracle.transform_array(b)
    if dtype in (np.float32, np.float64):
        same_zero = (a == 0) & (b == 0)
        lt = (a < b) | (same_zero & np.signbit(a) & ~np.signbit(b))
    else:
        lt = a < b
    assert np.array_equal(ca < cb, lt)


@pytest.mark.parametrize("dtype", KINDS)
@pytest.mark.parametrize("desc", [False, True])
def test_code_roundtrip(dtype, desc):
    a = _sample(dtype, 1 << 16, 13)
    u = _uint_view(dtype)
    structured = np.array([0, 1, 0x7FFFFFFF, 0x80000000, 0x80000001, 0xFFFFFFFF, 0x7F800000, 0xFF800000],
                          dtype=np.uint64)
    if np.dtype(dtype).itemsize == 8:
        structured = np.concatenate([structured, np.array(
            [0x7FFFFFFFFFFFFFFF, 0x8000000000000000, 0x8000000000000001, 0xFFFFFFFFFFFFFFFF,
             0x7FF0000000000000, 0xFFF0000000000000, 0x3FF0000000000000, 0xBFF0000000000000], dtype=np.uint64)])
    extra = structured.astype(u).view(dtype)
    a = np.concatenate([a, extra])
    back = oracle.inverse_array(oracle.transform_array(a, desc), dtype, desc)
    assert np.array_equal(back.view(u), a.view(u))


# --------------------------------------------------------------------------
# LSD radix sort
# --------------------------------------------------------------------------

def _uint_view(dtype):
    return np.uint64 if np.dtype(dtype).itemsize == 8 else np.uint32


def _sample(dtype, n, seed):
    seed = wl.seed_for(80, seed)
    if dtype == np.uint32:
        return wl.uniform_u32(n, seed)
    if dtype == np.int32:
        return wl.uniform_i32(n, seed)
    if dtype == np.float32:
        return wl.normal_mix_f32(n, seed)
    if dtype == np.int64:
        return wl.uniform_i64(n, seed)
    if dtype == np.float64:
        return wl.normal_mix_f64(n, seed)
    return wl.uniform_u64(n, seed)


def _few_distinct(dtype, n, seed, k=5):
    base = _sample(dtype, k, seed)
    idx = (wl.uniform_u32(n, wl.seed_for(81, seed)) % np.uint32(k)).astype(np.int64)
    return base[idx]


def _library_order(keys, descending, begin_bit=0, end_bit=None):
    """Stable order from numpy's stable sort on the native key (no oracle code)."""
    dtype = keys.dtype
    if dtype in (np.float32, np.float64):
        # value first; among the two zeros, -0.0 before +0.0
        pos_zero = (keys == 0) & ~np.signbit(keys)
        if descending:
            order = np.lexsort((~pos_zero, -keys.astype(np.float64)))
        else:
            order = np.lexsort((pos_zero, keys.astype(np.float64)))
        return order
    if end_bit is not None and (begin_bit, end_bit) != (0, keys.dtype.itemsize * 8):
        assert dtype in (np.uint32, np.uint64)
        w = end_bit - begin_bit
        k = (keys.astype(np.uint64) >> np.uint64(begin_bit)) & np.uint64((1 << w) - 1 if w < 64 else 2**64 - 1)
    else:
        k = keys
    if descending:
        if k.dtype in (np.int32, np.int64):
            k = ~k  # -k - 1: order reversed, no overflow at the minimum
        else:
            k = np.iinfo(k.dtype).max - k
    return np.argsort(k, kind="stable")


def _library_sorted_keys(keys, descending):
    return keys[_library_order(keys, descending)]


@pytest.mark.parametrize("dtype", KINDS)
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("n", [0, 1, 2, 33, 1000, 4099])
def test_lsd_matches_numpy_stable_sort(dtype, desc, n):
    for keys in (_sample(dtype, n, n), _few_distinct(dtype, n, n)):
        vals = np.arange(n, dtype=np.uint32)
        order = _library_order(keys, desc)
        ko, vo = oracle.sort_pairs(keys, vals, descending=desc)
        assert np.array_equal(vo, order.astype(np.uint32))
        u = _uint_view(dtype)
        assert np.array_equal(ko.view(u), keys[order].view(u))
        assert np.array_equal(oracle.sort_keys(keys, descending=desc).view(u), keys[order].view(u))


@pytest.mark.parametrize("dtype,rng_bits", [(np.uint32, [(0, 16), (3, 29), (8, 9), (0, 1), (31, 32), (5, 5)]),
                                            (np.uint64, [(0, 52), (17, 64), (60, 64), (0, 8)])])
@pytest.mark.parametrize("desc", [False, True])
def test_lsd_partial_bit_range(dtype, rng_bits, desc):
    keys = _sample(dtype, 3001, 21)
    for b, e in rng_bits:
        vals = np.arange(keys.size, dtype=np.uint32)
        order = _library_order(keys, desc, b, e)
        ko, vo = oracle.sort_pairs(keys, vals, b, e, descending=desc)
        assert np.array_equal(vo, order.astype(np.uint32)), (b, e)
        assert np.array_equal(ko, keys[order])


@pytest.mark.parametrize("n", range(0, 8))
def test_lsd_all_permutations_brute_force(n):
    for perm in itertools.permutations(range(n)):
        keys = np.array(perm, dtype=np.uint32) * np.uint32(0x01010101)
        assert oracle.sort_keys(keys).tolist() == sorted(keys.tolist())


def test_lsd_multisets_python_sorted():
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(0, 40))
        alphabet = rng.integers(0, 2**32, int(rng.integers(1, 6)), dtype=np.uint64).astype(np.uint32)
        keys = alphabet[rng.integers(0, alphabet.size, n)]
        vals = np.arange(n, dtype=np.uint32)
        want = sorted(range(n), key=lambda i: int(keys[i]))
        ko, vo = oracle.sort_pairs(keys, vals)
        assert vo.tolist() == want
        wantd = sorted(range(n), key=lambda i: int(keys[i]), reverse=True)  # stable in Python
        kd, vd = oracle.sort_pairs(keys, vals, descending=True)
        assert vd.tolist() == wantd


def test_lsd_composition_identity():
    # a [0,32) sort equals four stable byte sorts applied low to high ("GPU基数排序", §2)
    keys = _few_distinct(np.uint32, 5000, 3, k=300) ^ wl.uniform_u32(5000, 77) & np.uint32(0x0F0F0F0F)
    vals = np.arange(keys.size, dtype=np.uint32)
    k, v = keys, vals
    for b in (0, 8, 16, 24):
        k, v = oracle.sort_pairs(k, v, b, b + 8)
    ko, vo = oracle.sort_pairs(keys, vals, 0, 32)
    assert np.array_equal(k, ko) and np.array_equal(v, vo)
    # doing the bytes high to low (MSD order with stable passes) gives a different order in general
    k2, v2 = keys, vals
    for b in (24, 16, 8, 0):
        k2, v2 = oracle.sort_pairs(k2, v2, b, b + 8)
    assert not np.array_equal(k2, ko)


def test_digit_histograms_match_bincount():
    keys = wl.low_entropy_u32(10000, 9)
    h = oracle.digit_histograms(keys)
    for p in range(4):
        want = np.bincount((keys >> np.uint32(8 * p)) & np.uint32(255), minlength=256)
        assert np.array_equal(h[p], want)
    h16 = oracle.digit_histograms(keys, 3, 14)  # digits [3,11) and [11,14)
    assert np.array_equal(h16[0], np.bincount((keys >> np.uint32(3)) & np.uint32(255), minlength=256))
    assert np.array_equal(h16[1][:8], np.bincount((keys >> np.uint32(11)) & np.uint32(7), minlength=8))
    assert h16[1][8:].sum() == 0
    k64 = wl.priority_u64(5000, 4)
    h64 = oracle.digit_histograms(k64)
    assert h64.shape == (8, 256)
    assert h64[7][0] == 5000 and h64[6][16:].sum() == 0
    hd = oracle.digit_histograms(keys, descending=True)
    assert np.array_equal(hd[:, ::-1], h)


def test_in_place_call_matches():
    keys = wl.uniform_u32(1000, 1)
    want = oracle.sort_keys(keys)
    assert np.array_equal(want, np.sort(keys))


def test_float_sort_places_signed_zeros_and_infinities():
    keys = wl.normal_mix_f32(20000, 3)
    assert not np.isnan(keys).any()
    out = oracle.sort_keys(keys)
    assert np.isneginf(out[0]) and np.isposinf(out[-1])
    zeros = np.flatnonzero(out == 0)
    assert np.signbit(out[zeros[: (np.signbit(keys) & (keys == 0)).sum()]]).all()
    assert not np.signbit(out[zeros[(np.signbit(keys) & (keys == 0)).sum():]]).any()
    assert (out[1:] >= out[:-1]).all()


def test_workload_recipe_shapes():
    # the generators produce the advertised distributions (no sorting involved)
    n = 1 << 16
    f = wl.normal_mix_f32(n, 1)
    assert 0.04 < np.mean(f == 0) < 0.06
    assert 0.005 < np.mean(np.isinf(f)) < 0.015
    finite = f[np.isfinite(f) & (f != 0)]
    assert 900 < finite.std() < 1100
    le = wl.low_entropy_u32(n, 2)
    assert 0.1 < np.mean(le & np.uint32(1)) < 0.15
    a = wl.ascending_u32(n, 3)
    assert (np.diff(a.astype(np.int64)) >= 0).all()
    assert (wl.descending_u32(n, 3) == a[::-1]).all()
    p = wl.priority_u64(n, 4)
    assert (p >> np.uint64(52) == 0).all() and len(np.unique(p >> np.uint64(48))) == 16
    assert math.isclose(np.mean(wl.uniform_u32(n, 5).astype(np.float64)) / 2**32, 0.5, abs_tol=0.01)
    # counter-based: a slice equals the same draws of a longer stream
    assert np.array_equal(wl.splitmix64(7, 10), wl.splitmix64(7, 100)[:10])


def test_splitmix64_published_outputs():
    # first three outputs of SplitMix64 from state 0 (Vigna's reference splitmix64.c)
    assert [int(x) for x in wl.splitmix64(0, 3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                                      0x06C45D188009454F]


def test_torch_generator_draws_the_host_stream():
    torch = pytest.importorskip("torch")
    # the published first output of state 0, through the torch form (high 32 bits)
    assert int(wl.uniform_u32_torch(1, 0, "cpu").numpy().view(np.uint32)[0]) == 0xE220A839
    for n, chunk in ((1, 1 << 20), (100003, 4096), (1 << 20, 1 << 18)):
        seed = wl.seed_for(3, 20)
        got = wl.uniform_u32_torch(n, seed, "cpu", chunk=chunk).numpy().view(np.uint32)
        assert np.array_equal(got, wl.uniform_u32(n, seed))
