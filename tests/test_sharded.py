"""The multi-GPU sort's planning and exchange (sorting_lsd_radix_gb300.sharded).

CPU tests: the host planning functions on their own, then the whole sharded
sort on 2 and 4 gloo ranks (one process each, rendezvous on 127.0.0.1) with
the local steps run by the CPU oracle (tests/sharded_helpers.OracleOps).  The
concatenation of the ranks' outputs in rank order must equal the oracle's
stable sort of the concatenation of the shards, keys and values (values are
global input positions, so stability across ranks is checked too).

GPU test: the device steps of a multi-rank sort (digit histograms, the
partition pass, the local sort) for several virtual ranks run one after
another on one GPU through the C ABI, with the exchange done by slicing; the
result is checked against the oracle.  No kernels of different ranks ever
wait on one another.  The exchange path itself also runs on a one-rank NCCL
group, the rank acting as its own peer, so its collectives (histogram
all-gather, all-to-all-v of keys and values) run through NCCL on the GPU."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

from sorting_lsd_radix_gb300 import sharded  # noqa: E402
from tests.sharded_helpers import shard_keys  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _u(a):
    return a.view(np.uint64 if a.dtype.itemsize == 8 else np.uint32)


# ---------------------------------------------------------------------------
# host planning
# ---------------------------------------------------------------------------

def test_partition_digit_is_the_highest_varying_digit():
    h = np.zeros((4, 256), dtype=np.int64)
    h[3, 7] = 10  # top digit the same for all 10 keys
    h[2, 1], h[2, 9] = 4, 6
    h[1, 0] = 10
    h[0, 3], h[0, 4] = 5, 5
    assert sharded.partition_digit(h) == 2
    h2 = np.zeros((4, 256), dtype=np.int64)
    h2[:, 5] = 10
    assert sharded.partition_digit(h2) is None


def test_plan_ranges_balances_at_digit_boundaries():
    hist = np.full(256, 10, dtype=np.int64)  # 2560 keys, uniform digits
    b = sharded.plan_ranges(hist, np.array([640, 640, 640, 640]))
    assert b.tolist() == [0, 64, 128, 192, 256]
    skew = np.zeros(256, dtype=np.int64)
    skew[3], skew[200] = 900, 100  # two digit values only
    b = sharded.plan_ranges(skew, np.array([500, 500]))
    assert b[0] == 0 and b[2] == 256 and 4 <= b[1] <= 200  # the boundary falls between the two values
    # boundaries never decrease, even for targets far from any boundary
    b = sharded.plan_ranges(skew, np.array([1, 1, 998]))
    assert all(b[i] <= b[i + 1] for i in range(3))


def test_exchange_counts_sum_to_every_shard_and_every_receiver():
    rng = np.random.default_rng(1)
    local = rng.integers(0, 50, size=(3, 256))
    b = sharded.plan_ranges(local.sum(axis=0), local.sum(axis=1))
    c = sharded.exchange_counts(local, b)
    assert (c.sum(axis=1) == local.sum(axis=1)).all()
    recv = c.sum(axis=0)
    g = local.sum(axis=0)
    assert recv.tolist() == [int(g[b[r]:b[r + 1]].sum()) for r in range(3)]


# ---------------------------------------------------------------------------
# gloo ranks
# ---------------------------------------------------------------------------

WORKER = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import numpy as np, torch, torch.distributed as dist
from sorting_lsd_radix_gb300 import sharded
from tests.sharded_helpers import OracleOps, shard_keys
kind, sizes, desc, pairs, outdir = json.loads(sys.argv[2])
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", rank=rank, world_size=world)
keys = shard_keys(kind, rank, sizes[rank], 1)
vals = None
if pairs:
    vals = torch.from_numpy((np.arange(sizes[rank]) + sum(sizes[:rank])).astype(np.uint32))
k, v = sharded.sharded_sort(torch.from_numpy(keys), vals, descending=desc, ops=OracleOps())
np.save(os.path.join(outdir, f"k{rank}.npy"), k.numpy())
if v is not None:
    np.save(os.path.join(outdir, f"v{rank}.npy"), v.numpy())
dist.barrier()
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(tmp_path, kind, sizes, desc=False, pairs=False):
    world = len(sizes)
    port = _free_port()
    cfg = json.dumps([kind, sizes, desc, pairs, str(tmp_path)])
    procs = []
    for rank in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER, ROOT, cfg], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    for p in procs:
        _, err = p.communicate(timeout=300)
        assert p.returncode == 0, err
    keys = [np.load(tmp_path / f"k{r}.npy") for r in range(world)]
    vals = [np.load(tmp_path / f"v{r}.npy") for r in range(world)] if pairs else None
    return keys, vals


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("kind,desc", [("u32", False), ("f32", True), ("u64", False), ("i32", True),
                                       ("u32_low", False)])
def test_gloo_sharded_sort_keys(tmp_path, world, kind, desc):
    sizes = [30000 + 7919 * r for r in range(world)]
    out, _ = _run_ranks(tmp_path, kind, sizes, desc=desc)
    allin = np.concatenate([shard_keys(kind, r, sizes[r], 1) for r in range(world)])
    want = oracle.sort_keys(allin, descending=desc)
    got = np.concatenate(out)
    assert got.size == allin.size
    assert np.array_equal(_u(got), _u(want))
    # each rank's output is the matching slice of the global order
    off = 0
    for r in range(world):
        assert np.array_equal(_u(out[r]), _u(want[off:off + out[r].size]))
        off += out[r].size


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_sharded_sort_pairs_is_stable_across_ranks(tmp_path, world):
    sizes = [20011 + 3001 * r for r in range(world)]
    keys, vals = _run_ranks(tmp_path, "u32", sizes, pairs=True)
    allin = np.concatenate([shard_keys("u32", r, sizes[r], 1) for r in range(world)])
    wk, wv = oracle.sort_pairs(allin, np.arange(allin.size, dtype=np.uint32))
    assert np.array_equal(np.concatenate(keys), wk)
    assert np.array_equal(np.concatenate(vals), wv)  # ties in (rank, position) order


def test_gloo_all_equal_keys_stay_in_place(tmp_path):
    sizes = [1000, 2000]
    keys, vals = _run_ranks(tmp_path, "equal", sizes, pairs=True)
    assert [k.size for k in keys] == sizes
    assert np.array_equal(np.concatenate(vals), np.arange(3000, dtype=np.uint32))


# ---------------------------------------------------------------------------
# device steps on one GPU, several virtual ranks one after another
# ---------------------------------------------------------------------------

@pytest.mark.gpu
@pytest.mark.parametrize("kind,desc,pairs", [("u32", False, True), ("f32", True, False), ("u64", False, True)])
def test_device_steps_of_a_four_rank_sort(kind, desc, pairs):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sorting_lsd_radix_gb300 import build as gbuild
    gbuild.build()
    ops = sharded.DeviceOps()
    world = 4
    sizes = [70001 + 9973 * r for r in range(world)]
    shards = [shard_keys(kind, r, sizes[r], 2) for r in range(world)]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    dk = [torch.from_numpy(s).cuda() for s in shards]
    dv = [torch.arange(offs[r], offs[r + 1], dtype=torch.int64).to(torch.int32).view(torch.uint32).cuda()
          if pairs else None for r in range(world)]
    hists = np.stack([ops.digit_histograms(k, desc, None).cpu().numpy() for k in dk])
    for r in range(world):  # the histogram kernel against the oracle
        assert np.array_equal(hists[r], oracle.digit_histograms(shards[r], descending=desc).astype(np.int64))
    g = hists.sum(axis=0)
    p = sharded.partition_digit(g)
    bounds = sharded.plan_ranges(g[p], np.array(sizes))
    counts = sharded.exchange_counts(hists[:, p, :], bounds)
    parts = [ops.sort(dk[r], dv[r], 8 * p, 8 * p + 8, desc, None) for r in range(world)]
    for r in range(world):  # the partition pass against the oracle
        assert np.array_equal(_u(parts[r][0].cpu().numpy()), _u(oracle.sort_keys(shards[r], 8 * p, 8 * p + 8,
                                                                                   descending=desc)))
    outs_k, outs_v = [], []
    for dst in range(world):
        ks, vs = [], []
        for src in range(world):
            lo = int(counts[src, :dst].sum())
            ks.append(parts[src][0][lo:lo + int(counts[src, dst])])
            if pairs:
                vs.append(parts[src][1][lo:lo + int(counts[src, dst])])
        rk = torch.cat(ks)
        rv = torch.cat(vs) if pairs else None
        k, v = ops.sort(rk, rv, 0, 8 * rk.element_size(), desc, None)
        outs_k.append(k.cpu().numpy())
        if pairs:
            outs_v.append(v.cpu().numpy())
    allin = np.concatenate(shards)
    if pairs:
        wk, wv = oracle.sort_pairs(allin, np.arange(allin.size, dtype=np.uint32), descending=desc)
        assert np.array_equal(np.concatenate(outs_v), wv)
    else:
        wk = oracle.sort_keys(allin, descending=desc)
    assert np.array_equal(_u(np.concatenate(outs_k)), _u(wk))


@pytest.mark.gpu
@pytest.mark.parametrize("kind,desc,pairs", [("u32", False, True), ("f64", True, False), ("u64", False, False)])
def test_nccl_exchange_on_one_rank(kind, desc, pairs):
    """The exchange path on a one-rank NCCL group: the all-gather of the histograms and the
    all-to-all-v of keys and values go through NCCL with the rank as its own peer."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import torch.distributed as dist
    from sorting_lsd_radix_gb300 import build as gbuild
    gbuild.build()
    keys = shard_keys(kind, 0, 300007, 3)
    vals = np.arange(keys.size, dtype=np.uint32)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    try:
        k, v = sharded.sharded_sort(torch.from_numpy(keys).cuda(),
                                    torch.from_numpy(vals).cuda() if pairs else None,
                                    descending=desc, exchange_alone=True)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    if pairs:
        wk, wv = oracle.sort_pairs(keys, vals, descending=desc)
        assert np.array_equal(v.cpu().numpy(), wv)
    else:
        wk = oracle.sort_keys(keys, descending=desc)
    assert np.array_equal(_u(k.cpu().numpy()), _u(wk))


@pytest.mark.gpu
def test_sharded_segmented_sort_blocks():
    """Segments shard with no collective: each rank sorts its own consecutive block of segments.
    Without a process group the one rank's block is every segment."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sorting_lsd_radix_gb300 import build as gbuild
    gbuild.build()
    segs, seg_len = 37, 3000
    keys = shard_keys("u32", 0, segs * seg_len, 5)
    out, first = sharded.sharded_segmented_sort(torch.from_numpy(keys).cuda(), segs, seg_len, descending=True)
    assert first == 0 and out.numel() == keys.size
    assert np.array_equal(out.cpu().numpy(), oracle.segmented_sort(keys, segs, seg_len, descending=True))
