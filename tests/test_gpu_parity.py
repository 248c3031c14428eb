"""GPU parity: every entry point, through the C ABI, bit-exact against the oracle
on the same seeded inputs (keys compared as bit patterns, values exactly)."""
import numpy as np
import pytest

import oracle
from sorting_lsd_radix_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DTYPES = [np.uint32, np.int32, np.float32, np.uint64, np.int64, np.float64]


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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(t):
    return t.cpu().numpy()


def sample(dtype, n, seed):
    s = wl.seed_for(70, seed)
    if dtype == np.uint32:
        return wl.uniform_u32(n, s)
    if dtype == np.int32:
        return wl.uniform_i32(n, s)
    if dtype == np.float32:
        return wl.normal_mix_f32(n, s)
    if dtype == np.int64:
        return wl.uniform_i64(n, s)
    if dtype == np.float64:
        return wl.normal_mix_f64(n, s)
    return wl.uniform_u64(n, s)


def with_ties(dtype, n, seed, k=37):
    base = sample(dtype, k, seed + 1000)
    return base[(wl.uniform_u32(n, wl.seed_for(71, seed)) % np.uint32(k)).astype(np.int64)]


# Radix tile sizes of the launch shapes: 8192 keys (u32 keys and u32 pairs),
# 6144 (u64 keys), 5120 (u64 keys with u32 values, u32 keys with u64 values),
# 4096 (u64 keys with u64 values).  The sizes straddle each boundary, span
# several tiles with a ragged tail, and cross the bitonic/radix switch at 16384
# keys.
TILE32 = 8192
TILE64 = 6144
TILE64P = 5120
TILE64V64 = 4096
SIZES = [0, 1, 2, 31, 32, 33, 1023, TILE64P - 1, TILE64P, TILE64P + 1, 4095, 4096, 4097, TILE64 - 1, TILE64,
         TILE64 + 1, TILE32 - 1, TILE32, TILE32 + 1, 16383, 16384, 16385, 3 * TILE32 + 5, 5 * TILE64 + 3,
         7 * TILE64P + 9, (1 << 16) + 7, (1 << 20) + 3]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_sort_keys_full_range(g, dtype, desc, n):
    keys = sample(dtype, n, n)
    out, temp = g.gbs_sort_keys(_dev(keys), descending=desc, return_temp=True)
    assert np.array_equal(_u(_host(out)), _u(oracle.sort_keys(keys, descending=desc)))
    assert g.gbs_get_status(temp) == g.GBS_OK


def test_repeated_large_sorts_report_no_timeout(g):
    # many tiles per pass and repeated calls on one work buffer: every device
    # wait must end well inside its bound (a timeout would be recorded)
    n = (1 << 24) + 12345
    keys = wl.uniform_u32(n, wl.seed_for(2, 9))
    d = _dev(keys)
    out, temp = g.gbs_sort_keys(d, return_temp=True)
    for _ in range(8):
        g.gbs_sort_keys(d, keys_out=out, temp=temp)
        assert g.gbs_get_status(temp) == g.GBS_OK
    vals = torch.arange(n, dtype=torch.int32, device="cuda").view(torch.uint32) if hasattr(torch, "uint32") else None
    assert np.array_equal(_host(out), oracle.sort_keys(keys))
    if vals is not None:
        for _ in range(4):
            ko, vo, t2 = g.gbs_sort_pairs(d, vals, begin_bit=0, end_bit=32, return_temp=True)
            assert g.gbs_get_status(t2) == g.GBS_OK


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("n", [3, 1000, 16384, 16385, 50001])
def test_sort_pairs_with_ties_stable(g, dtype, desc, n):
    keys = with_ties(dtype, n, n)
    vals = np.arange(n, dtype=np.uint32)
    ko, vo = g.gbs_sort_pairs(_dev(keys), _dev(vals), descending=desc)
    ek, ev = oracle.sort_pairs(keys, vals, descending=desc)
    assert np.array_equal(_u(_host(ko)), _u(ek))
    assert np.array_equal(_host(vo), ev)


BIT_RANGES = {np.uint32: [(0, 16), (3, 29), (8, 9), (0, 1), (31, 32), (5, 5), (16, 32), (0, 24)],
              np.int32: [(0, 16), (20, 32)],
              np.float32: [(0, 8), (23, 32)],
              np.uint64: [(0, 52), (17, 64), (60, 64), (0, 8), (32, 64), (7, 7)],
              np.int64: [(0, 40), (40, 64)],
              np.float64: [(0, 8), (52, 64)]}


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("n", [3, 1000, 4097, 16385, 3 * TILE32 + 13])
def test_sort_pairs64_stable(g, dtype, desc, n):
    # 64-bit values follow the oracle's stable permutation (the oracle sorts (key, index) pairs)
    keys = with_ties(dtype, n, n + 3)
    vals = wl.uniform_u64(n, wl.seed_for(74, n))
    _, order = oracle.sort_pairs(keys, np.arange(n, dtype=np.uint32), descending=desc)
    ko, vo = g.gbs_sort_pairs(_dev(keys), _dev(vals), descending=desc)
    assert np.array_equal(_u(_host(ko)), _u(keys[order.astype(np.int64)]))
    assert np.array_equal(_host(vo), vals[order.astype(np.int64)])


@pytest.mark.parametrize("dtype", [np.uint32, np.uint64])
@pytest.mark.parametrize("bits", [(0, 16), (8, 8), (4, 28)])
def test_sort_pairs64_in_place_bit_ranges(g, dtype, bits):
    n = 2 * TILE32 + 77
    keys = with_ties(dtype, n, 19, k=500)
    vals = wl.uniform_u64(n, wl.seed_for(75, 1))
    _, order = oracle.sort_pairs(keys, np.arange(n, dtype=np.uint32), bits[0], bits[1])
    tk, tv = _dev(keys), _dev(vals)
    g.gbs_sort_pairs(tk, tv, keys_out=tk, vals_out=tv, begin_bit=bits[0], end_bit=bits[1])
    assert np.array_equal(_host(tk), keys[order.astype(np.int64)])
    assert np.array_equal(_host(tv), vals[order.astype(np.int64)])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("desc", [False, True])
def test_partial_bit_ranges_pairs(g, dtype, desc):
    n = 3 * TILE32 + 11
    keys = sample(dtype, n, 5)
    vals = np.arange(n, dtype=np.uint32)
    for b, e in BIT_RANGES[dtype]:
        ko, vo = g.gbs_sort_pairs(_dev(keys), _dev(vals), begin_bit=b, end_bit=e, descending=desc)
        ek, ev = oracle.sort_pairs(keys, vals, b, e, descending=desc)
        assert np.array_equal(_u(_host(ko)), _u(ek)), (b, e)
        assert np.array_equal(_host(vo), ev), (b, e)
        kk = g.gbs_sort_keys(_dev(keys), begin_bit=b, end_bit=e, descending=desc)
        assert np.array_equal(_u(_host(kk)), _u(ek)), (b, e)


@pytest.mark.parametrize("dist", list(wl.DISTRIBUTIONS_U32))
@pytest.mark.parametrize("desc", [False, True])
def test_distributions_u32(g, dist, desc):
    n = (1 << 20) + 77
    keys = wl.DISTRIBUTIONS_U32[dist](n, wl.seed_for(2, 3))
    got = _host(g.gbs_sort_keys(_dev(keys), descending=desc))
    assert np.array_equal(got, oracle.sort_keys(keys, descending=desc))
    vals = np.arange(n, dtype=np.uint32)
    ko, vo = g.gbs_sort_pairs(_dev(keys), _dev(vals), begin_bit=0, end_bit=16, descending=desc)
    ek, ev = oracle.sort_pairs(keys, vals, 0, 16, descending=desc)
    assert np.array_equal(_host(ko), ek) and np.array_equal(_host(vo), ev)


@pytest.mark.parametrize("dtype", [np.uint32, np.uint64])
@pytest.mark.parametrize("n", [5000, 3 * TILE32 + 1, 200003])
@pytest.mark.parametrize("bits", [(0, 32), (0, 8), (4, 20), (9, 9)])
def test_in_place(g, dtype, n, bits):
    keys = with_ties(dtype, n, 7, k=300) if dtype == np.uint32 else sample(dtype, n, 7) & np.uint64(0xFFFF00FF)
    vals = np.arange(n, dtype=np.uint32)
    tk, tv = _dev(keys), _dev(vals)
    g.gbs_sort_pairs(tk, tv, keys_out=tk, vals_out=tv, begin_bit=bits[0], end_bit=bits[1])
    ek, ev = oracle.sort_pairs(keys, vals, bits[0], bits[1])
    assert np.array_equal(_host(tk), ek) and np.array_equal(_host(tv), ev)
    tk2 = _dev(keys)
    g.gbs_sort_keys(tk2, keys_out=tk2, begin_bit=bits[0], end_bit=bits[1], descending=True)
    assert np.array_equal(_host(tk2), oracle.sort_keys(keys, bits[0], bits[1], descending=True))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [0, 1, 1000, 16385, 3 * TILE32 + 7])
@pytest.mark.parametrize("pinned", [True, False])
def test_sort_keys_host_buffers(g, dtype, n, pinned):
    keys = sample(dtype, n, n + 11)
    h_in = torch.from_numpy(np.ascontiguousarray(keys))
    if pinned:
        h_in = h_in.pin_memory()
    out, temp = g.gbs_sort_keys_host(h_in, descending=(n % 2 == 1), return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK  # synchronises the stream
    assert not out.is_cuda
    assert np.array_equal(_u(out.numpy()), _u(oracle.sort_keys(keys, descending=(n % 2 == 1))))
    assert np.array_equal(_u(h_in.numpy()), _u(keys))  # input untouched


@pytest.mark.parametrize("bits", [(0, 32), (4, 20), (8, 8)])
def test_sort_keys_host_in_place_bit_ranges(g, bits):
    n = 2 * TILE32 + 13
    keys = with_ties(np.uint32, n, 91)
    h = torch.from_numpy(keys.copy()).pin_memory()
    out, temp = g.gbs_sort_keys_host(h, h, begin_bit=bits[0], end_bit=bits[1], return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK
    assert out.data_ptr() == h.data_ptr()
    assert np.array_equal(h.numpy(), oracle.sort_keys(keys, bits[0], bits[1]))


BATCH_SIZES = [5000, 0, 2 * TILE32 + 13, 1, 16385, 3, 100003, 16384, 2 * TILE32 + 13]


@pytest.mark.parametrize("dtype", [np.uint32, np.float32, np.int64, np.float64])
@pytest.mark.parametrize("descending", [False, True])
def test_sort_keys_host_batch(g, dtype, descending):
    """Arrays of mixed sizes (empty, one key, the one-CTA bitonic path, several ragged radix tiles) sorted
    by one batch call; more arrays than device key buffers, so buffers are reused; one array in place."""
    keys = [sample(dtype, n, 300 + i) if i % 3 else with_ties(dtype, n, 300 + i) for i, n in enumerate(BATCH_SIZES)]
    h_in = [torch.from_numpy(np.ascontiguousarray(k)).pin_memory() for k in keys]
    h_out = [torch.empty_like(t).pin_memory() for t in h_in]
    h_out[2] = h_in[2]  # in place
    out, temp = g.gbs_sort_keys_host_batch(h_in, h_out, descending=descending, return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK  # synchronises the stream
    for i, k in enumerate(keys):
        assert out[i].data_ptr() == h_out[i].data_ptr()
        assert np.array_equal(_u(out[i].numpy()), _u(oracle.sort_keys(k, descending=descending))), i
        if i != 2:
            assert np.array_equal(_u(h_in[i].numpy()), _u(k))  # inputs untouched


@pytest.mark.parametrize("bits", [(4, 20), (8, 8), (0, 32)])
def test_sort_keys_host_batch_bit_ranges_and_reused_work_buffer(g, bits):
    sizes = [3 * TILE32 + 7, 40000, 10]
    keys = [with_ties(np.uint32, n, 500 + n) for n in sizes]
    h_in = [torch.from_numpy(k.copy()).pin_memory() for k in keys]
    out, temp = g.gbs_sort_keys_host_batch(h_in, begin_bit=bits[0], end_bit=bits[1], return_temp=True)
    out2 = g.gbs_sort_keys_host_batch(h_in, begin_bit=bits[0], end_bit=bits[1], temp=temp)
    assert g.gbs_get_status(temp) == g.GBS_OK
    for i, k in enumerate(keys):
        want = oracle.sort_keys(k, bits[0], bits[1])
        assert np.array_equal(out[i].numpy(), want) and np.array_equal(out2[i].numpy(), want)


def test_sort_keys_host_batch_empty_and_ordering(g):
    # an empty batch clears the header and enqueues nothing else
    _, temp = g.gbs_sort_keys_host_batch([], return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK
    # the copies wait for work enqueued on the stream before the call: the input is written by a device
    # copy just before, and the output is read right after the stream (and nothing else) is synchronised
    n = 2 * TILE32 + 5
    keys = wl.uniform_u32(n, 77)
    src = _dev(keys.view(np.int32))
    h = torch.empty(n, dtype=torch.int32).pin_memory()
    h.copy_(src, non_blocking=True)  # device-to-host copy enqueued on the current stream
    out = g.gbs_sort_keys_host_batch([h], key_type=g.GBS_U32)
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(out[0].numpy().view(np.uint32), oracle.sort_keys(keys))


def test_all_passes_trivial_and_skipped_passes(g):
    n = 3 * TILE32 + 9
    eq = wl.all_equal_u32(n, 1)
    assert np.array_equal(_host(g.gbs_sort_keys(_dev(eq), begin_bit=0, end_bit=32)), eq)
    vals = np.arange(n, dtype=np.uint32)
    ko, vo = g.gbs_sort_pairs(_dev(eq), _dev(vals))
    assert np.array_equal(_host(vo), vals)
    # only the middle byte varies: passes 0, 1 and 3 are trivial
    k = (wl.uniform_u32(n, 2) & np.uint32(0x00FF0000)) | np.uint32(0x12003456)
    ko, vo = g.gbs_sort_pairs(_dev(k), _dev(vals))
    assert g.gbs_debug_last_launch_count() == 5  # histogram + four pass kernels
    ek, ev = oracle.sort_pairs(k, vals)
    assert np.array_equal(_host(ko), ek) and np.array_equal(_host(vo), ev)
    # u64 keys whose top byte is zero (7 active passes of 8)
    k64 = wl.priority_u64(n, 3)
    ko, vo = g.gbs_sort_pairs(_dev(k64), _dev(vals))
    ek, ev = oracle.sort_pairs(k64, vals)
    assert np.array_equal(_host(ko), ek) and np.array_equal(_host(vo), ev)


def test_unaligned_pointers_use_plain_loads(g):
    n = 5 * TILE32 + 3
    base = wl.uniform_u32(n + 1, 9)
    t = _dev(base)
    view_in = t[1:]  # 4-byte aligned, not 16-byte aligned
    out = torch.empty(n + 1, dtype=torch.uint32, device="cuda")[1:]
    g.gbs_sort_keys(view_in, keys_out=out, begin_bit=0, end_bit=24)
    assert np.array_equal(_host(out), oracle.sort_keys(base[1:], 0, 24))


def test_concurrent_streams_with_separate_work_buffers(g):
    # independent calls on two streams overlap on the GPU; each has its own work buffer
    n1, n2 = 3 * TILE32 + 101, 5 * TILE64 + 7
    k1 = sample(np.uint32, n1, 301)
    k2 = sample(np.float64, n2, 302)
    v1 = np.arange(n1, dtype=np.uint32)
    d1, d2, dv1 = _dev(k1), _dev(k2), _dev(v1)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        o1, ov1, t1 = g.gbs_sort_pairs(d1, dv1, descending=True, return_temp=True, stream=s1)
    with torch.cuda.stream(s2):
        o2, t2 = g.gbs_sort_keys(d2, return_temp=True, stream=s2)
    for _ in range(5):
        g.gbs_sort_pairs(d1, dv1, keys_out=o1, vals_out=ov1, descending=True, temp=t1, stream=s1)
        g.gbs_sort_keys(d2, keys_out=o2, temp=t2, stream=s2)
    s1.synchronize()
    s2.synchronize()
    ek, ev = oracle.sort_pairs(k1, v1, descending=True)
    assert np.array_equal(_host(o1), ek) and np.array_equal(_host(ov1), ev)
    assert np.array_equal(_u(_host(o2)), _u(oracle.sort_keys(k2)))
    assert g.gbs_get_status(t1, stream=s1) == g.GBS_OK and g.gbs_get_status(t2, stream=s2) == g.GBS_OK


@pytest.mark.parametrize("n", [5000, 3 * TILE32 + 5])
def test_sort_captured_in_cuda_graph(g, n):
    # every entry point only enqueues work on the stream, so a call can be captured once and
    # replayed on new contents of the same buffers
    d_in = _dev(sample(np.uint32, n, 401))
    d_out = torch.empty_like(d_in)
    v_in = _dev(np.arange(n, dtype=np.uint32))
    v_out = torch.empty_like(v_in)
    _, temp = g.gbs_sort_keys(d_in, keys_out=d_out, return_temp=True)           # warm-up: kernel set-up
    _, _, ptemp = g.gbs_sort_pairs(d_in, v_in, keys_out=d_out, vals_out=v_out, descending=True, return_temp=True)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.gbs_sort_keys(d_in, keys_out=d_out, temp=temp)
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pgraph):
        g.gbs_sort_pairs(d_in, v_in, keys_out=d_out, vals_out=v_out, descending=True, temp=ptemp)
    for seed in (402, 403):
        keys = with_ties(np.uint32, n, seed)
        d_in.copy_(_dev(keys))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_host(d_out), oracle.sort_keys(keys))
        pgraph.replay()
        torch.cuda.synchronize()
        ek, ev = oracle.sort_pairs(keys, np.arange(n, dtype=np.uint32), descending=True)
        assert np.array_equal(_host(d_out), ek) and np.array_equal(_host(v_out), ev)
    assert g.gbs_get_status(temp) == g.GBS_OK and g.gbs_get_status(ptemp) == g.GBS_OK


def test_temp_reuse_across_calls(g):
    n = 100000
    a = wl.uniform_u32(n, 11)
    b = wl.low_entropy_u32(n, 12)
    _, temp = g.gbs_sort_keys(_dev(a), return_temp=True, begin_bit=0, end_bit=20)
    for keys in (b, a, b):
        got = _host(g.gbs_sort_keys(_dev(keys), temp=temp, begin_bit=0, end_bit=20))
        assert np.array_equal(got, oracle.sort_keys(keys, 0, 20))
    assert g.gbs_get_status(temp) == g.GBS_OK


SEG_LENS = [1, 2, 3, 5, 16, 31, 32, 33, 100, 255, 256, 1000, 1024, 1025, 2048, 4096, 8191, 8192, 16383, 16384]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("seg_len", SEG_LENS)
def test_segmented_sort(g, dtype, seg_len):
    segs = max(3, min(300, (1 << 18) // seg_len))
    keys = sample(dtype, segs * seg_len, seg_len)
    if seg_len % 3 == 0:
        keys = with_ties(dtype, segs * seg_len, seg_len)
    for desc in (False, True):
        got = _host(g.gbs_segmented_sort(_dev(keys), segs, seg_len, descending=desc))
        assert np.array_equal(_u(got), _u(oracle.segmented_sort(keys, segs, seg_len, descending=desc))), desc


SEG_MIX = [0, 1, 2, 3, 5, 17, 100, 255, 256, 1000, 1023, 1024, 1025, 2047, 4097, 8191, 16383, 16384, 16385,
           20000, 70001, 0, 7, 300, 3000]


R11_SIZES = [16385, 4095 * 5, 4096 * 7, 8192 * 3 + 1, 8192 * 5, 100003, (1 << 20) + 9]
R11_RANGES = {np.uint32: [(0, 32), (0, 22), (5, 27), (21, 32)], np.int32: [(0, 32)], np.float32: [(0, 32), (9, 31)],
              np.uint64: [(0, 64), (0, 33), (40, 64)], np.int64: [(0, 64)], np.float64: [(0, 64), (11, 55)]}


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", R11_SIZES)
def test_radix11_prototype(g, dtype, n):
    """The 11-bit-digit prototype (2048 digit values per pass) sorts exactly like the 8-bit path:
    every key type, both orders, partial bit ranges, ties, in place."""
    keys = sample(dtype, n, n % 89) if n % 2 else with_ties(dtype, n, n % 89)
    g.gbs_debug_set_radix_bits(11)
    try:
        for b, e in R11_RANGES[dtype]:
            for desc in (False, True):
                out, temp = g.gbs_sort_keys(_dev(keys), begin_bit=b, end_bit=e, descending=desc, return_temp=True)
                assert g.gbs_get_status(temp) == g.GBS_OK
                assert np.array_equal(_u(_host(out)), _u(oracle.sort_keys(keys, b, e, descending=desc))), (b, e, desc)
        t = _dev(keys)
        g.gbs_sort_keys(t, keys_out=t)  # in place (an odd number of passes for 32-bit keys)
        assert np.array_equal(_u(_host(t)), _u(oracle.sort_keys(keys)))
    finally:
        g.gbs_debug_set_radix_bits(8)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [16385, 100003, 1 << 21])
def test_msd_bitonic_hybrid(g, dtype, n):
    """MSD radix passes over the top 16 code bits, then a bitonic sort of every bucket: the
    result is the full-width sort (ties are identical keys, so order among them is invisible)."""
    keys = sample(dtype, n, n % 97)
    for desc in (False, True):
        got = _host(g.gbs_sort_keys_msd_bitonic(_dev(keys), descending=desc))
        assert np.array_equal(_u(got), _u(oracle.sort_keys(keys, descending=desc))), desc


def test_msd_bitonic_hybrid_skewed_buckets(g):
    # the AND of three draws leaves most top-16-bit prefixes near zero: buckets far above 2^14
    # keys take the radix path, the rest the bitonic network; many buckets are empty
    keys = wl.low_entropy_u32(1 << 20, wl.seed_for(72, 1))
    t = _dev(keys)
    out, temp = g.gbs_sort_keys_msd_bitonic(t, return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK
    assert np.array_equal(_host(out), oracle.sort_keys(keys))
    g.gbs_sort_keys_msd_bitonic(t, keys_out=t, temp=temp)  # in place
    assert np.array_equal(_host(t), oracle.sort_keys(keys))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("seg_len", [16385, 40000, 65537])
def test_segmented_sort_long_segments(g, dtype, seg_len):
    """Fixed-length segments above one CTA's network take the radix path, segment by segment."""
    segs = 3
    keys = sample(dtype, segs * seg_len, seg_len) if seg_len != 40000 else with_ties(dtype, segs * seg_len, seg_len)
    for desc in (False, True):
        got = _host(g.gbs_segmented_sort(_dev(keys), segs, seg_len, descending=desc))
        want = np.concatenate([oracle.sort_keys(keys[i * seg_len:(i + 1) * seg_len], descending=desc)
                               for i in range(segs)])
        assert np.array_equal(_u(got), _u(want)), desc
    t = _dev(keys)
    out, temp = g.gbs_segmented_sort(t, segs, seg_len, keys_out=t, return_temp=True)  # in place
    assert g.gbs_get_status(temp) == g.GBS_OK
    want = np.concatenate([oracle.sort_keys(keys[i * seg_len:(i + 1) * seg_len]) for i in range(segs)])
    assert np.array_equal(_u(_host(t)), _u(want))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("desc", [False, True])
@pytest.mark.parametrize("in_place", [False, True])
def test_segmented_sort_offsets(g, dtype, desc, in_place):
    # lengths of every class (0, 1, 2^l and its neighbours, past 2^14), a leading and a trailing gap
    extra = (wl.uniform_u32(40, wl.seed_for(72, 1)) % np.uint32(600)).astype(np.int64)
    lens = np.array(SEG_MIX + extra.tolist(), dtype=np.int64)
    offs = np.concatenate([[7], 7 + np.cumsum(lens)])
    n = int(offs[-1]) + 9
    keys = with_ties(dtype, n, 73, k=5000) if desc else sample(dtype, n, 73)
    tin = _dev(keys)
    if in_place:
        out = g.gbs_segmented_sort_offsets(tin, offs, keys_out=tin, descending=desc)
    else:
        out = g.gbs_segmented_sort_offsets(tin, offs, descending=desc)  # keys_out starts as a copy
    got = _host(out)
    u = _u
    for s_, e_ in zip(offs[:-1], offs[1:]):
        want = oracle.sort_keys(keys[s_:e_], descending=desc)
        assert np.array_equal(u(got[s_:e_]), u(want)), (s_, e_ - s_)
    assert np.array_equal(u(got[:7]), u(keys[:7])) and np.array_equal(u(got[offs[-1]:]), u(keys[offs[-1]:]))
    if not in_place:
        assert np.array_equal(u(_host(tin)), u(keys))


def test_segmented_offsets_empty_and_status(g):
    t = _dev(wl.uniform_u32(100, 3))
    out, temp = g.gbs_segmented_sort_offsets(t, [0], return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK
    out, temp = g.gbs_segmented_sort_offsets(t, [10, 10, 10, 90], return_temp=True)
    assert g.gbs_get_status(temp) == g.GBS_OK
    h = _host(t)
    assert np.array_equal(_host(out)[10:90], np.sort(h[10:90])) and np.array_equal(_host(out)[:10], h[:10])


def test_segmented_zero_one_principle_exhaustive(g):
    # every 0-1 pattern of 16 keys, one per segment ("并行排序" §1.2, 0-1 principle)
    pats = wl.zero_one_patterns(16)
    got = _host(g.gbs_segmented_sort(_dev(pats.reshape(-1)), pats.shape[0], 16)).reshape(pats.shape)
    ones = pats.sum(axis=1)
    want = (np.arange(16)[None, :] >= (16 - ones)[:, None]).astype(np.uint32)
    assert np.array_equal(got, want)
    assert np.array_equal(got.reshape(-1), oracle.segmented_sort(pats.reshape(-1), pats.shape[0], 16))


def test_segmented_in_place_and_empty(g):
    keys = sample(np.uint32, 64 * 700, 3)
    t = _dev(keys)
    g.gbs_segmented_sort(t, 64, 700, keys_out=t, descending=True)
    assert np.array_equal(_host(t), oracle.segmented_sort(keys, 64, 700, descending=True))
    e = torch.empty(0, dtype=torch.uint32, device="cuda")
    assert g.gbs_segmented_sort(e, 0, 100).numel() == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("desc", [False, True])
def test_digit_histograms(g, dtype, desc):
    n = 200001
    keys = with_ties(dtype, n, 4) if dtype == np.float32 else sample(dtype, n, 4)
    for b, e in [(0, 8 * keys.dtype.itemsize), (3, 29), (0, 16)]:
        got = _host(g.gbs_digit_histograms(_dev(keys), b, e, descending=desc)).astype(np.int64)
        assert np.array_equal(got, oracle.digit_histograms(keys, b, e, descending=desc).astype(np.int64))


def test_worked_example_on_gpu(g):
    src = np.array([4, 2, 7, 1, 8, 3, 6, 5], dtype=np.uint32)  # kwkr.cn notes §2.2
    assert _host(g.gbs_sort_keys(_dev(src))).tolist() == [1, 2, 3, 4, 5, 6, 7, 8]
    assert _host(g.gbs_segmented_sort(_dev(src), 1, 8)).tolist() == [1, 2, 3, 4, 5, 6, 7, 8]


def test_float_special_values(g):
    vals = np.array([np.inf, -0.0, 0.0, -np.inf, 1.0, -1.0, np.float32(1e-45), -np.float32(1e-45), 3.4e38,
                     -3.4e38] * 3000, dtype=np.float32)
    for desc in (False, True):
        for n in (30, 30000):
            got = _host(g.gbs_sort_keys(_dev(vals[:n]), descending=desc))
            assert np.array_equal(got.view(np.uint32), oracle.sort_keys(vals[:n], descending=desc).view(np.uint32))


def test_double_special_values(g):
    vals = np.array([np.inf, -0.0, 0.0, -np.inf, 1.0, -1.0, 5e-324, -5e-324, 1.7e308, -1.7e308,
                     np.nextafter(1.0, 2.0), np.nextafter(-1.0, -2.0)] * 3000, dtype=np.float64)
    for desc in (False, True):
        for n in (36, 36000):
            got = _host(g.gbs_sort_keys(_dev(vals[:n]), descending=desc))
            assert np.array_equal(got.view(np.uint64), oracle.sort_keys(vals[:n], descending=desc).view(np.uint64))
        seg = _host(g.gbs_segmented_sort(_dev(vals[:36 * 512]), 36, 512, descending=desc))
        want = oracle.segmented_sort(vals[:36 * 512], 36, 512, descending=desc)
        assert np.array_equal(seg.view(np.uint64), want.view(np.uint64))


def test_int64_extremes(g):
    ext = np.array([-2**63, 2**63 - 1, -1, 0, 1, -2**62, 2**62] * 5000, dtype=np.int64)
    for desc in (False, True):
        got = _host(g.gbs_sort_keys(_dev(ext), descending=desc))
        assert np.array_equal(got, oracle.sort_keys(ext, descending=desc))
