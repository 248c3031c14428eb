"""Benchmark: device-wide LSD radix sort of 1e8 uniform uint32 keys on GB300.

One step = one gbs_sort_keys call (full 32-bit range: the upfront histogram
kernel plus four one-sweep digit passes) over 1e8 keys already resident in
HBM.  The input (400 MB) is larger than L2, so no L2 flush is done between
steps.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gbsort|reference]

--impl reference times the CPU oracle (single-threaded serial LSD radix sort)
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sorting_lsd_radix_gb300 import workloads as wl  # noqa: E402

N_KEYS = 100_000_000
SEED = wl.seed_for(3, 0)
METRIC = "uint32 keys sorted/s at n=1e8; achieved HBM GB/s vs GB300 peak"
UNIT = "keys/s"
WORKLOAD = "sort_keys u32 ascending, bits [0,32), n=1e8 i.i.d. uniform keys (SplitMix64)"
FALLBACK_HBM_GBS = 6800.0
PASS_KERNEL_SOURCES = ["sorting_lsd_radix_gb300/csrc/radix_impl.cuh", "sorting_lsd_radix_gb300/csrc/common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "onesweep_pass_u32_traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gbsort", choices=["gbsort", "reference"])
    ap.add_argument("--n", type=int, default=N_KEYS)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="headline", choices=["headline"] + sorted(SECONDARY),
                    help="headline: the benchmark line; others: the remaining configurations, one JSON line each")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


NOMINAL_HBM_GBS = 2 * 3996e6 * 8192 / 8 / 1e9  # 3996 MHz double data rate on an 8192-bit bus


def theoretical_hbm_gbs():
    """Pin-rate bound of the HBM: 2 x memory clock x bus width, from the device's own
    attributes where torch exposes them, else the nominal GB300 figures."""
    try:
        import torch
        pr = torch.cuda.get_device_properties(torch.cuda.current_device())
        gbs = 2.0 * pr.memory_clock_rate * 1e3 * pr.memory_bus_width / 8 / 1e9
        if 1000.0 < gbs < 20000.0:
            return gbs, f"device attributes: {pr.memory_clock_rate / 1e3:.0f} MHz x {pr.memory_bus_width}-bit x 2"
    except Exception:
        pass
    return NOMINAL_HBM_GBS, "nominal: 3996 MHz x 8192-bit x 2"


def source_hash():
    h = hashlib.sha256()
    for rel in PASS_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(n):
    """DRAM bytes per pass-kernel launch from the committed ncu record (profiles/*.json), scaled to
    n keys (traffic grows in proportion to n); None if absent or taken on a different kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        if rec["source_sha256_16"] != source_hash():
            return None
        return float(rec["dram_bytes_per_launch"]) * n / float(rec["n"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_sm_clock_hz(gpu_index=0):
    """The GPU's maximum SM clock from nvidia-smi; 2070 MHz (GB300) if it cannot be read."""
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10).stdout
        return float(out.strip().splitlines()[0]) * 1e6
    except Exception:
        return 2070e6


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, dist, device):
    """The largest of every rank's value (one all-reduce); the value itself on one rank.  device: where
    the process group's backend keeps tensors ("cuda" for NCCL, "cpu" for gloo)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, n_per_rank, ms_per_step):
    """Whole-job keys/s: every rank sorts its own n keys per step; the step time is the slowest rank's."""
    return world * n_per_rank / (ms_per_step / 1e3)


def cpu_baseline(n_total, seconds=10.0):
    """The oracle as it stands, single-threaded, on a bounded slice of the workload."""
    import oracle
    sample_n = min(n_total, 1 << 24)
    keys = wl.uniform_u32(sample_n, SEED)
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        t0 = time.perf_counter()
        oracle.sort_keys(keys)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end or len(times) >= 20:
            break
    med = statistics.median(times)
    return {"value": sample_n / med, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {sample_n} keys of the workload (same generator and seed), serial LSD radix sort, "
                      f"median of {len(times)} runs",
            "library_sort": library_sort_baseline(keys)}


def library_sort_baseline(keys, seconds=5.0):
    """Side baseline: the host's library comparison sort (numpy.sort, default kind) on one
    core, on the same sample as the oracle."""
    import numpy as np
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        t0 = time.perf_counter()
        np.sort(keys)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end or len(times) >= 20:
            break
    med = statistics.median(times)
    return {"value": keys.size / med, "unit": UNIT, "cores": 1, "kind": "numpy.sort (library sort, one thread)",
            "sample": f"the same {keys.size} keys, median of {len(times)} runs"}


def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    import oracle
    sample_n = min(args.n, 1 << 23)
    keys = wl.uniform_u32(sample_n, SEED)
    for _ in range(args.warmup):
        oracle.sort_keys(keys)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sort_keys(keys)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = sample_n / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n": args.n, "step_sample_keys": sample_n},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"first {sample_n} keys of the workload per step, serial LSD radix sort"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gbsort(args):
    import torch
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from sorting_lsd_radix_gb300 import build as gbuild
    gbuild.build()
    from sorting_lsd_radix_gb300 import gbsort, sharded

    n = args.n
    host = wl.uniform_u32(n, SEED + rank)
    d_in = torch.from_numpy(host).cuda()
    stream = torch.cuda.current_stream()
    if world == 1:
        d_out = torch.empty_like(d_in)
        _, temp = gbsort.gbs_sort_keys(d_in, d_out, return_temp=True)

        def step():
            gbsort.gbs_sort_keys(d_in, d_out, temp=temp)
            return d_out
    else:
        # one array of world * n keys held in shards: the sample-sort exchange across the GPUs
        def step():
            return sharded.sharded_sort(d_in)[0]
    out = step()
    torch.cuda.synchronize()
    launches = gbsort.gbs_debug_last_launch_count()  # kernels of the step's last sorting call

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timing: K steps between two events ----------------
    for _ in range(args.warmup):
        out = step()
    # per-kernel events of every timed step's (last) sorting call: histogram and 4 passes
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(launches + 1)] for _ in range(args.steps)]
    for evs in events:  # torch creates the CUDA event on first record
        for e in evs:
            e.record(stream)
    barrier()
    sampler = ClockSampler(local)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(args.steps):
        gbsort.gbs_debug_set_timing_events(events[s])
        out = step()
    stop.record(stream)
    gbsort.gbs_debug_set_timing_events(None)
    barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(start.elapsed_time(stop), dist, "cuda")
    ms_per_step = ms / args.steps
    status = gbsort.gbs_get_status(temp) if world == 1 else gbsort.GBS_OK
    per_kernel = np.array([[ev[i].elapsed_time(ev[i + 1]) for i in range(launches)] for ev in events])

    # correctness spot check of the timed output (full checks are in the tests): sorted, and for
    # the sharded sort every rank's last key is at most the next rank's first key
    out_host = out.cpu().numpy()
    ok = bool((out_host[1:] >= out_host[:-1]).all()) and status == gbsort.GBS_OK
    if dist is not None:
        edge = torch.tensor([int(out_host[0]) if out_host.size else 2**32, int(out_host[-1]) if out_host.size else -1],
                            dtype=torch.int64, device="cuda")
        edges = [torch.empty_like(edge) for _ in range(world)]
        dist.all_gather(edges, edge)
        e = [t.cpu().tolist() for t in edges]
        ok = ok and all(e[r][1] <= e[r + 1][0] for r in range(world - 1) if e[r][1] >= 0 and e[r + 1][0] < 2**32)
        total = torch.tensor([out_host.size], dtype=torch.int64, device="cuda")
        dist.all_reduce(total)
        ok = ok and int(total.item()) == world * n

    # ---- end to end: the C-ABI host-buffer entry point (copy in, sort, copy out)
    e2e = None
    if not args.no_e2e and world > 1:
        # the sharded sort from host memory: each rank copies its shard in, the GPUs sort the whole
        # array together, each rank copies its part of the result back
        h_in = torch.from_numpy(host).pin_memory()

        def e2e_step():
            part = sharded.sharded_sort(h_in.cuda(non_blocking=True))[0]
            return part.cpu()
        for _ in range(2):
            e2e_step()
        barrier()
        k = max(3, min(args.steps, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            hv = e2e_step()
        e1.record(stream)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1) / k, dist, "cuda")
        hvn = hv.numpy()
        ok = ok and bool((hvn[1:] >= hvn[:-1]).all())
        e2e = {"value": job_throughput(world, n, ems), "unit": UNIT, "h2d_bytes_per_step": 4 * n,
               "d2h_bytes_per_step": 4 * int(hvn.size), "ms_per_step": ems,
               "api": "sorting_lsd_radix_gb300.sharded.sharded_sort on a copy of the host shard"}
    elif not args.no_e2e:
        h_in = torch.from_numpy(host).pin_memory()
        h_out = torch.empty_like(h_in).pin_memory()
        _, htemp = gbsort.gbs_sort_keys_host(h_in, h_out, temp=None, return_temp=True)
        for _ in range(2):
            gbsort.gbs_sort_keys_host(h_in, h_out, temp=htemp)
        barrier()
        k = max(3, min(args.steps, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            gbsort.gbs_sort_keys_host(h_in, h_out, temp=htemp)
        e1.record(stream)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1) / k, dist, "cuda")
        ok = ok and gbsort.gbs_get_status(htemp) == gbsort.GBS_OK
        hv = h_out.numpy()
        ok = ok and bool((hv[1:] >= hv[:-1]).all())
        e2e = {"value": job_throughput(world, n, ems), "unit": UNIT, "h2d_bytes_per_step": 4 * n,
               "d2h_bytes_per_step": 4 * n, "ms_per_step": ems}

        # A stream of host sorts through the batch entry point: kb steps in one call, each step still
        # copying its 1e8 keys in and its result out (inputs repeat; two output buffers alternate).
        # The call overlaps step i's sort with step i + 1's copy in and step i - 1's copy out, so the
        # two directions of the host link run together.  This throughput is the reported e2e value;
        # the one-at-a-time figure above is kept beside it.
        outs = [h_out, torch.empty_like(h_in).pin_memory()]
        _, btemp = gbsort.gbs_sort_keys_host_batch([h_in, h_in], outs, return_temp=True)
        kb = 32  # arrays per call: the pipeline's fill and drain (about one step) are spread over 32
        ins_b, outs_b = [h_in] * kb, [outs[i % 2] for i in range(kb)]
        gbsort.gbs_sort_keys_host_batch(ins_b, outs_b, temp=btemp)  # warm-up
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gbsort.gbs_sort_keys_host_batch(ins_b, outs_b, temp=btemp)
        e1.record(stream)
        barrier()
        pms = max_over_ranks(e0.elapsed_time(e1) / kb, dist, "cuda")
        ok = ok and gbsort.gbs_get_status(btemp) == gbsort.GBS_OK
        for j in range(2):
            hv = outs[j].numpy()
            ok = ok and bool((hv[1:] >= hv[:-1]).all())
        e2e = {"value": job_throughput(world, n, pms), "unit": UNIT, "h2d_bytes_per_step": 4 * n,
               "d2h_bytes_per_step": 4 * n, "ms_per_step": pms, "steps_per_call": kb,
               "api": f"gbs_sort_keys_host_batch ({kb} host arrays of n keys per call, pinned buffers; "
                      f"copies in and out overlapped with the sorts)",
               "one_step_at_a_time": {"value": e2e["value"], "unit": UNIT, "ms_per_step": ems,
                                      "api": "gbs_sort_keys_host, one call per step"}}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peak, peak_kind = peaks()
    theo, theo_src = theoretical_hbm_gbs()
    # dominant kernel: the one-sweep digit pass (kernels 1..4 of each call)
    pass_ms = per_kernel[:, 1:5].mean()
    hist_ms = per_kernel[:, 0].mean()
    alg_pass = 8.0 * n  # 4-byte key read + 4-byte key write per key
    achieved = alg_pass / (pass_ms / 1e3) / 1e9
    traffic = recorded_traffic(n)
    alg_total = 36.0 * n  # histogram read (4n) + 4 passes x 8n
    cpu = None if args.no_cpu_baseline else cpu_baseline(n)
    line = {
        "metric": METRIC, "value": job_throughput(world, n, ms_per_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "n": n, "key_type": "u32", "begin_bit": 0, "end_bit": 32,
                   "seed": SEED, "l2": "input 400 MB > L2; no flush between steps",
                   "parallelism": (f"one array of {world} x {n} keys sharded over {world} GPUs: digit histograms, "
                                   f"one partition pass, one all-to-all-v exchange (NCCL), local radix sort"
                                   if world > 1 else "one GPU")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": f"onesweep_pass_kernel<u32,keys,tile={gbsort.gbs_debug_radix_tile_keys(4)}>",
                     "peak_kind": f"{peak_kind} hbm_gbs",
                     "theoretical_peak": theo, "theoretical_source": theo_src,
                     "frac_of_theoretical": achieved / theo,
                     "algorithmic_bytes_per_launch": alg_pass, "avg_launch_ms": pass_ms},
        "whole_sort": {"achieved_gbs": alg_total / (ms_per_step / 1e3) / 1e9,
                       "frac_of_peak": alg_total / (ms_per_step / 1e3) / 1e9 / peak,
                       "frac_of_theoretical": alg_total / (ms_per_step / 1e3) / 1e9 / theo,
                       "algorithmic_bytes": alg_total, "histogram_ms": hist_ms, "pass_ms": pass_ms,
                       "kernel_ms": per_kernel.mean(axis=0).tolist()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": (launches if world == 1 else launches + 3) * args.steps,
        "clocks": clocks,
        "check": {"sorted": ok, "status": gbsort.status_string(status)},
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# Secondary workloads (the other configurations; informative lines, not the
# benchmark line).  Each entry: description, builder(n) -> (call, n_keys,
# algorithmic bytes per call, dominant-kernel algorithmic bytes per launch,
# dominant-kernel launch indices, extra fields).
# ---------------------------------------------------------------------------

def _active_passes(gbsort, d_keys, begin, end, desc):
    """Digit passes whose digit is not the same for every key (a pass with one digit value moves
    nothing and is skipped by the sort), from the library's own upfront-histogram kernel."""
    hist = gbsort.gbs_digit_histograms(d_keys, begin_bit=begin, end_bit=end, descending=desc).cpu().numpy()
    return [p for p in range(hist.shape[0]) if np.count_nonzero(hist[p]) > 1]


def _sec_radix_keys(gen, n_default, key_type, begin=0, end=None, desc=False, radix_bits=8):
    def build(gbsort, torch, n=None):
        n = n or n_default
        gbsort.gbs_debug_set_radix_bits(radix_bits)
        keys = gen(n)
        d = torch.from_numpy(keys).cuda()
        o = torch.empty_like(d)
        s = keys.itemsize
        stop = end if end is not None else 8 * s
        passes = (stop - begin + 7) // 8
        active = _active_passes(gbsort, d, begin, stop, desc)
        # the sort call last: the caller reads its launch count
        _, temp = gbsort.gbs_sort_keys(d, o, begin_bit=begin, end_bit=end, descending=desc, return_temp=True)
        # histogram read + one read and one write per active pass (all trivial: the last pass
        # launch copies the keys once)
        alg = s * n + max(len(active), 1) * 2 * s * n
        dom = [1 + p for p in active] if active else [passes]
        call = lambda: gbsort.gbs_sort_keys(d, o, begin_bit=begin, end_bit=end, descending=desc, temp=temp)
        extra = {"active_passes": len(active), "oracle_sample": (keys, begin, stop, desc)}
        if radix_bits != 8:
            # 11-bit digits: ceil(bits / 11) passes; all of them active on these workloads
            passes = (stop - begin + radix_bits - 1) // radix_bits
            alg = s * n + passes * 2 * s * n
            dom = list(range(1, passes + 1))
            extra.update({"active_passes": passes, "radix_bits": radix_bits})
        return call, temp, n, alg, 2 * s * n, dom, extra
    return build


def _sec_radix_graph(n):
    """The u32 sort captured once in a CUDA graph and replayed (no per-call host work)."""
    def build(gbsort, torch):
        keys = wl.uniform_u32(n, wl.seed_for(1, 0))
        d = torch.from_numpy(keys).cuda()
        o = torch.empty_like(d)
        _, temp = gbsort.gbs_sort_keys(d, o, return_temp=True)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            gbsort.gbs_sort_keys(d, o, temp=temp)
        gbsort.gbs_sort_keys(d, o, temp=temp)  # leaves the launch count of one call for the timing events
        return graph.replay, temp, n, 36 * n, 8 * n, [], {"graph": True}
    return build


def _sec_pairs_u64(n_default):
    def build(gbsort, torch, n=None):
        n = n or n_default
        keys = wl.priority_u64(n, wl.seed_for(4, 0))
        d = torch.from_numpy(keys).cuda()
        v = torch.arange(n, dtype=torch.int32, device="cuda").view(torch.uint32)
        ko, vo = torch.empty_like(d), torch.empty_like(v)
        _, _, temp = gbsort.gbs_sort_pairs(d, v, ko, vo, return_temp=True)
        call = lambda: gbsort.gbs_sort_pairs(d, v, ko, vo, temp=temp)
        # bits 56..63 are zero: 7 active passes of 8 (the eighth returns at once)
        return call, temp, n, 8 * n + 7 * 24 * n, 24 * n, list(range(1, 8)), {"active_passes": 7}
    return build


def _sec_segmented(segs, seg_len):
    def build(gbsort, torch):
        keys = wl.uniform_u32(segs * seg_len, wl.seed_for(2, 0))
        d = torch.from_numpy(keys).cuda()
        o = torch.empty_like(d)
        call = lambda: gbsort.gbs_segmented_sort(d, segs, seg_len, keys_out=o)
        call()
        p = (seg_len - 1).bit_length()
        comps = segs * (1 << p) // 2 * p * (p + 1) // 2
        n = segs * seg_len
        return call, None, n, 8 * n, 8 * n, [0], {"comparators_per_call": comps}
    return build


def _sec_segmented_var(num_segments, max_len):
    def build(gbsort, torch):
        lens = (wl.uniform_u32(num_segments, wl.seed_for(2, 3)) % np.uint32(max_len) + 1).astype(np.int64)
        offs = np.concatenate([[0], np.cumsum(lens)])
        n = int(offs[-1])
        keys = wl.uniform_u32(n, wl.seed_for(2, 4))
        d = torch.from_numpy(keys).cuda()
        o = torch.empty_like(d)
        _, temp = gbsort.gbs_segmented_sort_offsets(d, offs, keys_out=o, return_temp=True)
        call = lambda: gbsort.gbs_segmented_sort_offsets(d, offs, keys_out=o, temp=temp)
        launches = gbsort.gbs_debug_last_launch_count()
        return call, temp, n, 8 * n, 8 * n, list(range(launches)), {"segments": num_segments,
                                                                      "length_classes": launches,
                                                                      "sum_dominant": True}
    return build


def _sec_msd_bitonic(n_default):
    """The hybrid prototype: MSD radix passes over the top 16 bits, then a bitonic sort per bucket."""
    def build(gbsort, torch, n=None):
        n = n or n_default
        keys = wl.uniform_u32(n, SEED)
        d = torch.from_numpy(keys).cuda()
        o = torch.empty_like(d)
        _, temp = gbsort.gbs_sort_keys_msd_bitonic(d, o, return_temp=True)
        call = lambda: gbsort.gbs_sort_keys_msd_bitonic(d, o, temp=temp)
        # two MSD passes (histogram read + 2 x (read + write)), the boundary scan (one read) and the
        # bitonic finish (one read and one write); timed as whole calls (the call synchronises once
        # for its host-side bucket plan, and its kernels are several library calls)
        return call, temp, n, 4 * n + 2 * 8 * n + 4 * n + 8 * n, 8 * n, [], \
            {"whole_call": True, "hybrid": "MSD 16 bits + bitonic per bucket"}
    return build


SECONDARY = {
    "u32_2p20": ("sort_keys u32 n=2^20 uniform (L2-resident: launch-latency bound, roofline not meaningful)",
                 _sec_radix_keys(lambda n: wl.uniform_u32(n, wl.seed_for(1, 0)), 1 << 20, "u32")),
    "u32_2p20_graph": ("sort_keys u32 n=2^20 uniform, captured in a CUDA graph and replayed",
                       _sec_radix_graph(1 << 20)),
    "u32_1e8_low_entropy": ("sort_keys u32 n=1e8, AND of three uniform draws",
                            _sec_radix_keys(lambda n: wl.low_entropy_u32(n, wl.seed_for(3, 1)), N_KEYS, "u32")),
    "u32_1e8_sorted": ("sort_keys u32 n=1e8, already ascending",
                       _sec_radix_keys(lambda n: wl.ascending_u32(n, wl.seed_for(3, 1)), N_KEYS, "u32")),
    "u32_1e8_reverse": ("sort_keys u32 n=1e8, descending input",
                        _sec_radix_keys(lambda n: wl.descending_u32(n, wl.seed_for(3, 1)), N_KEYS, "u32")),
    "u32_1e8_all_equal": ("sort_keys u32 n=1e8, all keys equal (every pass trivial: histogram + copy)",
                          _sec_radix_keys(lambda n: wl.all_equal_u32(n, wl.seed_for(3, 1)), N_KEYS, "u32")),
    "u32_1e8_msd_bitonic": ("sort_keys u32 n=1e8 uniform by the hybrid prototype: MSD radix over the top 16 bits, "
                            "then a bitonic sort of each of the 65536 buckets", _sec_msd_bitonic(N_KEYS)),
    "u32_1e8_radix11": ("sort_keys u32 n=1e8 uniform with the 11-bit-digit prototype (3 passes)",
                        _sec_radix_keys(lambda n: wl.uniform_u32(n, SEED), N_KEYS, "u32", radix_bits=11)),
    "i64_2p27_radix11": ("sort_keys i64 n=2^27 uniform with the 11-bit-digit prototype (6 passes)",
                         _sec_radix_keys(lambda n: wl.uniform_i64(n, wl.seed_for(6, 1)), 1 << 27, "i64",
                                         radix_bits=11)),
    "f64_2p27_radix11": ("sort_keys f64 n=2^27 N(0,1000) with signed zeros and infinities, 11-bit-digit prototype",
                         _sec_radix_keys(lambda n: wl.normal_mix_f64(n, wl.seed_for(6, 0)), 1 << 27, "f64",
                                         radix_bits=11)),
    "u32_2p30": ("sort_keys u32 n=2^30 uniform (4 GiB; from 2^29 keys on the look-back status words are 64-bit)",
                 _sec_radix_keys(lambda n: wl.uniform_u32(n, wl.seed_for(3, 2)), 1 << 30, "u32")),
    "u32_1e8_bits0_16": ("sort_keys u32 n=1e8 uniform, bits [0,16)",
                         _sec_radix_keys(lambda n: wl.uniform_u32(n, SEED), N_KEYS, "u32", 0, 16)),
    "f32_2p28": ("sort_keys f32 n=2^28, N(0,1000) with signed zeros and infinities",
                 _sec_radix_keys(lambda n: wl.normal_mix_f32(n, wl.seed_for(5, 0)), 1 << 28, "f32")),
    "f32_2p28_desc": ("sort_keys f32 n=2^28 descending",
                      _sec_radix_keys(lambda n: wl.normal_mix_f32(n, wl.seed_for(5, 0)), 1 << 28, "f32",
                                      desc=True)),
    "f64_2p27": ("sort_keys f64 n=2^27, N(0,1000) with signed zeros and infinities",
                 _sec_radix_keys(lambda n: wl.normal_mix_f64(n, wl.seed_for(6, 0)), 1 << 27, "f64")),
    "i64_2p27": ("sort_keys i64 n=2^27 uniform", _sec_radix_keys(lambda n: wl.uniform_i64(n, wl.seed_for(6, 1)),
                                                                  1 << 27, "i64")),
    "i32_2p28": ("sort_keys i32 n=2^28 uniform", _sec_radix_keys(lambda n: wl.uniform_i32(n, wl.seed_for(5, 1)),
                                                                 1 << 28, "i32")),
    "pairs_u64_2p27": ("sort_pairs u64 keys (4-bit priority << 48 | 48-bit field) + u32 index values, n=2^27",
                       _sec_pairs_u64(1 << 27)),
    "seg_16384x1024": ("segmented_sort u32, 16384 segments x 1024 keys", _sec_segmented(16384, 1024)),
    "seg_4096x16384": ("segmented_sort u32, 4096 segments x 16384 keys", _sec_segmented(4096, 16384)),
    "segvar_16384x1to2048": ("segmented_sort_offsets u32, 16384 segments of 1..2048 keys (uniform lengths)",
                             _sec_segmented_var(16384, 2048)),
}


def secondary_cpu_baseline(keys, begin, end, desc, seconds=10.0):
    """The oracle, single-threaded, on the first (up to) 2^22 keys of a secondary workload."""
    import oracle
    sample = np.ascontiguousarray(keys[: 1 << 22])
    times = []
    t_end = time.perf_counter() + seconds
    while True:
        t0 = time.perf_counter()
        oracle.sort_keys(sample, begin, end, descending=desc)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end or len(times) >= 5:
            break
    med = statistics.median(times)
    return {"value": sample.size / med, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {sample.size} keys of the workload, median of {len(times)} runs"}


def run_secondary(args):
    import torch
    torch.cuda.set_device(0)
    from sorting_lsd_radix_gb300 import build as gbuild
    gbuild.build()
    from sorting_lsd_radix_gb300 import gbsort
    desc, builder = SECONDARY[args.workload]
    # --n resizes the radix-sort workloads (a small case of the same distribution, e.g. for ncu)
    if args.n != N_KEYS and "n" in builder.__code__.co_varnames[:builder.__code__.co_argcount]:
        call, temp, n, alg_bytes, dom_bytes, dom_idx, extra = builder(gbsort, torch, args.n)
    else:
        call, temp, n, alg_bytes, dom_bytes, dom_idx, extra = builder(gbsort, torch)
    torch.cuda.synchronize()
    # a replayed CUDA graph bypasses the library's per-kernel timing hook: time whole calls only
    launches = 0 if (extra.get("graph") or extra.pop("whole_call", False)) else gbsort.gbs_debug_last_launch_count()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        call()
    steps = max(args.steps // 10, 5)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(launches + 1)] for _ in range(steps)]
    for evs in events:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in range(steps):
        gbsort.gbs_debug_set_timing_events(events[s_])
        call()
    e1.record(stream)
    gbsort.gbs_debug_set_timing_events(None)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    per_kernel = (np.array([[ev[i].elapsed_time(ev[i + 1]) for i in range(launches)] for ev in events]).mean(axis=0)
                  if launches else np.zeros(0))
    # the dominant figure is one launch's time, or all listed launches together (several kernels
    # sharing one job, e.g. one bitonic launch per segment-length class); the whole call when the
    # kernels are not timed one by one
    if not dom_idx:
        dom_ms = ms
    else:
        dom_ms = float(per_kernel[dom_idx].sum() if extra.pop("sum_dominant", False) else per_kernel[dom_idx].mean())
    peak, peak_kind = peaks()
    theo, _ = theoretical_hbm_gbs()
    line = {"workload": args.workload, "description": desc, "n": n, "ms_per_call": ms,
            "keys_per_s": n / (ms / 1e3), "algorithmic_bytes": alg_bytes,
            "achieved_gbs": alg_bytes / (ms / 1e3) / 1e9, "frac_of_peak": alg_bytes / (ms / 1e3) / 1e9 / peak,
            "dominant_kernel_ms": dom_ms, "dominant_kernel_gbs": dom_bytes / (dom_ms / 1e3) / 1e9,
            "dominant_kernel_frac": dom_bytes / (dom_ms / 1e3) / 1e9 / peak, "peak_gbs": peak,
            "peak_kind": f"{peak_kind} hbm_gbs", "theoretical_peak_gbs": theo,
            "frac_of_theoretical": alg_bytes / (ms / 1e3) / 1e9 / theo,
            "kernel_ms": per_kernel.tolist(), "launches": launches}
    if "comparators_per_call" in extra:
        line["comparators_per_s"] = extra["comparators_per_call"] / (ms / 1e3)
        # ALU roofline of the bitonic network: a compare-exchange is a min, a max and the
        # direction's complement (3 logic-pipe ops per pair of keys); the logic pipe retires 2 warp
        # instructions per clock per SM (64 lane ops)
        props = torch.cuda.get_device_properties(0)
        sm_clock_hz = max_sm_clock_hz()
        alu_peak = props.multi_processor_count * 64 * sm_clock_hz / 3
        kernel_ms = float(per_kernel.sum()) if launches else ms
        line["alu_roofline"] = {"bound": "alu", "achieved": extra["comparators_per_call"] / (kernel_ms / 1e3),
                                "peak": alu_peak, "unit": "compare-exchanges/s",
                                "frac": extra["comparators_per_call"] / (kernel_ms / 1e3) / alu_peak,
                                "peak_basis": f"{props.multi_processor_count} SMs x 64 logic-pipe lane ops per clock "
                                              f"x {sm_clock_hz / 1e9:.2f} GHz (maximum SM clock) / 3 ops per "
                                              f"compare-exchange"}
    sample = extra.pop("oracle_sample", None)
    line.update({k: v for k, v in extra.items() if k != "comparators_per_call"})
    if temp is not None:
        line["status"] = gbsort.status_string(gbsort.gbs_get_status(temp))
    if sample is not None and not args.no_cpu_baseline:
        line["cpu_baseline"] = secondary_cpu_baseline(*sample)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "headline":
        run_secondary(args)
    else:
        run_gbsort(args)


if __name__ == "__main__":
    main()
