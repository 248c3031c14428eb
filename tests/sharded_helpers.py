"""Test-only stand-ins for the sharded sort's local steps.

OracleOps runs each rank's local steps (digit histograms, stable sort by a bit
range) with the CPU oracle on CPU tensors, so that the product's planning and
exchange logic (sorting_lsd_radix_gb300.sharded) can run on gloo CPU ranks
without a GPU.  Test infrastructure only."""
import numpy as np
import torch

import oracle


class OracleOps:
    def digit_histograms(self, keys, descending, key_type):
        h = oracle.digit_histograms(keys.numpy(), descending=descending)
        return torch.from_numpy(h.astype(np.int64))

    def sort(self, keys, vals, begin_bit, end_bit, descending, key_type):
        k = keys.numpy()
        if vals is None:
            return torch.from_numpy(oracle.sort_keys(k, begin_bit, end_bit, descending=descending)), None
        ko, vo = oracle.sort_pairs(k, vals.numpy(), begin_bit, end_bit, descending=descending)
        return torch.from_numpy(ko), torch.from_numpy(vo)


def shard_keys(kind, rank, n, seed):
    """A rank's shard for the multi-rank tests: sizes differ per rank and keys repeat across ranks
    (ties whose order the stable global sort fixes by rank, then position)."""
    from sorting_lsd_radix_gb300 import workloads as wl
    s = wl.seed_for(80 + rank, seed)
    if kind == "u32":
        k = wl.uniform_u32(n, s) % np.uint32(5000)  # many ties, within and across ranks
    elif kind == "u32_low":
        k = wl.low_entropy_u32(n, s)
    elif kind == "f32":
        k = wl.normal_mix_f32(n, s)
    elif kind == "i32":
        k = wl.uniform_i32(n, s)
    elif kind == "u64":
        k = wl.priority_u64(n, s)  # bits 56..63 zero: the partition digit is the next one down
    elif kind == "f64":
        k = wl.normal_mix_f64(n, s)
    elif kind == "equal":
        k = np.full(n, 0xDEADBEEF, dtype=np.uint32)
    else:
        raise ValueError(kind)
    return np.ascontiguousarray(k)
