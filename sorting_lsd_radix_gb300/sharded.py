"""Sort one array held in shards across the ranks of a process group (one GPU per rank).

The pages' distributed method is sample sort with one exchange step
("并行排序：从归并网络到 GPU 双调排序" §7.1-7.3: choose splitters, bucket every
key by them, exchange the buckets with an all-to-all-v, sort locally).  Here
the splitters are digit boundaries:

1. every rank counts the digits of its shard (the upfront histogram kernel,
   all digit positions in one read) and the ranks all-gather those counts;
2. the partition digit is the highest digit position whose global histogram
   holds more than one value (every higher digit is the same for all keys, so
   ordering by this digit orders by the key code); each rank is given a
   contiguous range of its values, chosen so that the ranks' output sizes come
   as close as digit granularity allows to their input sizes.  Every rank
   computes the same plan from the same gathered counts, and from them its own
   send and receive counts, with no further collective;
3. each rank groups its keys by destination with one stable radix pass over the
   partition digit (the pass kernel);
4. one all-to-all-v moves the groups (NCCL on GPUs);
5. each rank sorts what it received (the full radix sort).

Output: rank r holds the r-th contiguous part of the globally sorted keys; in
rank order the parts are the stable sort of the concatenation of the shards in
rank order.  Ties keep (source rank, source position) order because every
local step is stable and the received pieces are concatenated in source-rank
order.  When every digit is the same for all keys, the concatenation of the
shards is already the stable order and each rank keeps its shard.

Every step on the keys runs in the library's kernels (`DeviceOps`); the
collectives are torch.distributed's.  The planning works on the 256-bin
counts only.  `ops` can be replaced so that the planning and exchange logic
runs on CPU ranks (gloo) in tests.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import gbsort


class DeviceOps:
    """The library's kernels on the current CUDA device."""

    def digit_histograms(self, keys: torch.Tensor, descending: bool, key_type: int | None) -> torch.Tensor:
        """Counts of every 8-bit digit position of the keys' codes, shape (key bits / 8, 256)."""
        return gbsort.gbs_digit_histograms(keys, descending=descending, key_type=key_type).to(torch.int64)

    def sort(self, keys: torch.Tensor, vals: torch.Tensor | None, begin_bit: int, end_bit: int,
             descending: bool, key_type: int | None):
        """Stable sort of keys (and values) by the code bits [begin_bit, end_bit)."""
        if vals is None:
            return gbsort.gbs_sort_keys(keys, begin_bit=begin_bit, end_bit=end_bit, descending=descending,
                                        key_type=key_type), None
        return gbsort.gbs_sort_pairs(keys, vals, begin_bit=begin_bit, end_bit=end_bit, descending=descending,
                                     key_type=key_type)


def partition_digit(global_hist: np.ndarray) -> int | None:
    """Highest digit position whose global histogram has more than one non-empty bin (None: every
    digit is the same for all keys)."""
    for p in range(global_hist.shape[0] - 1, -1, -1):
        if np.count_nonzero(global_hist[p]) > 1:
            return p
    return None


def plan_ranges(global_digit_hist: np.ndarray, targets: np.ndarray) -> np.ndarray:
    """Digit boundaries b[0] = 0 <= b[1] <= ... <= b[G] = 256: rank r receives the digit values
    [b[r], b[r+1]).  Boundary r is the digit boundary whose global key count before it is
    closest to the target position sum(targets[:r]) (the earliest such boundary on a tie)."""
    g = len(targets)
    cum = np.concatenate([[0], np.cumsum(global_digit_hist.astype(np.int64))])  # keys below each boundary
    pos = np.concatenate([[0], np.cumsum(np.asarray(targets, dtype=np.int64))])
    b = np.zeros(g + 1, dtype=np.int64)
    b[g] = 256
    for r in range(1, g):
        b[r] = max(int(np.argmin(np.abs(cum - pos[r]))), int(b[r - 1]))
    return b


def exchange_counts(local_hists: np.ndarray, bounds: np.ndarray) -> np.ndarray:
    """counts[src, dst]: keys rank src sends to rank dst, from every rank's partition-digit
    histogram (local_hists[src, digit]) and the digit ranges."""
    g = local_hists.shape[0]
    counts = np.zeros((g, g), dtype=np.int64)
    for dst in range(g):
        counts[:, dst] = local_hists[:, bounds[dst]:bounds[dst + 1]].sum(axis=1)
    return counts


def _wire(t: torch.Tensor) -> torch.Tensor:
    """The same bytes as a signed integer tensor, a type every backend exchanges."""
    return t.view(torch.int64 if t.element_size() == 8 else torch.int32)


def sharded_sort(keys: torch.Tensor, vals: torch.Tensor | None = None, descending: bool = False,
                 key_type: int | None = None, group=None, ops=None, exchange_alone: bool = False):
    """Globally sorts the shards held by the ranks of `group` (every rank calls this with its own
    shard; shards may differ in size).  Returns this rank's part of the sorted keys (and the values
    that travel with them): (keys, vals).  keys: 4- or 8-byte key tensor of any gbsort key type;
    vals: optional 4- or 8-byte values, moved with their keys (stable).  A group of one rank sorts
    locally, unless exchange_alone is set: then every step of the exchange runs with the rank as its
    own peer (the collectives included), which checks that path on a single GPU."""
    ops = ops or DeviceOps()
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if world == 1 and not exchange_alone:
        return ops.sort(keys, vals, 0, 8 * keys.element_size(), descending, key_type)

    # 1. digit counts of every rank
    hist = ops.digit_histograms(keys, descending, key_type)  # (P, 256) int64 on the keys' device
    gathered = [torch.empty_like(hist) for _ in range(world)]
    dist.all_gather(gathered, hist, group=group)
    local_hists = np.stack([h.cpu().numpy() for h in gathered])  # (G, P, 256)
    sizes = local_hists[:, 0, :].sum(axis=1)
    global_hist = local_hists.sum(axis=0)

    # 2. the plan (identical on every rank)
    p = partition_digit(global_hist)
    if p is None:  # every key has the same code: the shards in rank order are already sorted
        return keys.clone(), (None if vals is None else vals.clone())
    bounds = plan_ranges(global_hist[p], sizes)
    counts = exchange_counts(local_hists[:, p, :], bounds)

    # 3. group this shard's keys by destination: one stable pass over the partition digit
    part_k, part_v = ops.sort(keys, vals, 8 * p, 8 * p + 8, descending, key_type)

    # 4. one all-to-all-v
    send = [int(c) for c in counts[rank]]
    recv = [int(c) for c in counts[:, rank]]
    out_k = torch.empty(sum(recv), dtype=keys.dtype, device=keys.device)
    dist.all_to_all_single(_wire(out_k), _wire(part_k), output_split_sizes=recv, input_split_sizes=send,
                           group=group)
    out_v = None
    if vals is not None:
        out_v = torch.empty(sum(recv), dtype=vals.dtype, device=vals.device)
        dist.all_to_all_single(_wire(out_v), _wire(part_v), output_split_sizes=recv, input_split_sizes=send,
                               group=group)

    # 5. local sort of the received keys (full width)
    return ops.sort(out_k, out_v, 0, 8 * keys.element_size(), descending, key_type)


def sharded_segmented_sort(keys: torch.Tensor, num_segments: int, segment_len: int, descending: bool = False,
                           key_type: int | None = None, group=None):
    """Segmented sort of the segments [first, last) of this rank's share: the segments are
    independent, so every rank sorts its own consecutive block of them and no collective is
    needed.  keys holds all num_segments * segment_len keys on every rank; returns this rank's
    block of sorted segments and the index of its first segment."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    first = num_segments * rank // world
    last = num_segments * (rank + 1) // world
    part = keys[first * segment_len:last * segment_len]
    return gbsort.gbs_segmented_sort(part, last - first, segment_len, descending=descending,
                                     key_type=key_type), first
