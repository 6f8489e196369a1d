"""Benchmark: batched row-wise top-k + flat row gather on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                    [--no-per-workload] [--profile [--sorted-value]] [--profile-extra pair|block]

One step = one pass of the whole path over one batch of the workload: the
fused top-k + gather launch (sel_topk_gather) for the gather workloads, the
top-k launch (sel_topk) for the others.  Inputs are seeded synthetic data of
the workload's shape (no dataset), resident in HBM before timing starts; L2
is flushed (a 256 MiB write) before every timed step and the flush is not
timed.  Each step is timed with CUDA events on the launching stream.

Prints ONE JSON line on rank 0.  The default workload is the fp32 sampling
top-k on logits[256, 131072], k = 4096: the 128K-wide rows the top-k's
bandwidth target is quoted on.  Besides the contract's keys the line carries:
  per_workload      all five named workloads: flushed and warm-L2 step times,
                    the top-k alone (topk_only_*: for the gather workloads the
                    same selection without the fused gather, its own bytes and
                    fraction of peak), and the step with value-ordered output;
  pair_gather       the two-key gather (1024 x 512 positions, d 128 + 512);
  block_candidates  the block-level candidate chain with its gather;
  cpu_baseline      the oracle single-threaded, and row-parallel over the
                    host's cores (`row_parallel`).

--impl reference times the CPU oracle (the plain full-sort definition) on a
bounded sample of the same workload, on the host cores.

Profiling modes (short runs for ncu): --profile [--sorted-value] runs only the
warm-up and timed steps of --workload; --profile-extra pair|block runs only
the two-key gather or the block-level chain.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402

METRIC = "top-k effective HBM GB/s (fraction of GB300 peak) and rows/s per config, 1 GPU"
DEFAULT_WORKLOAD = "sampling_f32_256x131072_k4096_nan"
FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------
# algorithmic bytes (what the method must move; re-reads are not counted)
# ----------------------------------------------------------------------------

def valid_lengths(w) -> np.ndarray:
    if w["row_end"] is None:
        return np.full(w["rows"], w["cols"], dtype=np.int64)
    return np.clip(w["row_end"].astype(np.int64), 0, w["cols"])


def topk_bytes(w) -> int:
    """Read every valid element of rows with n > k, write k indices (and k values) per row."""
    e = syn.elem_bytes(w["dtype"])
    ib = 8 if w["idx_dtype"] == "i64" else 4
    n = valid_lengths(w)
    read = int(n[n > w["k"]].sum()) * e
    write = w["rows"] * w["k"] * (ib + (e if w["want_values"] else 0))
    return read + write


def gather_bytes(w, fused: bool) -> int:
    """The key + gathered rows written (+ the index read when not fused).  The whole key stands in
    for the unique key rows read: exact up to 2 rows on the 2048-key workload, an overcount of
    9.4 MB (3.2 MB of 12.6 MB are read; 0.5% of the step's bytes) on the 64-level one."""
    if w.get("key") is None:
        return 0
    key_bytes = w["b"] * w["comp_len"] * w["d"] * 2
    out = w["rows"] * w["n_gather"] * w["d"] * 2
    idx_read = 0 if fused else w["rows"] * w["n_gather"] * 4
    return key_bytes + out + idx_read


def step_bytes(w) -> int:
    return topk_bytes(w) + gather_bytes(w, fused=True)


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.tsv")
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth; fractions of it are reported beside the measured peak


def kernel_source_hash() -> str:
    """Short hash of the selection and gather kernels' source: a stored DRAM traffic figure is used only
    while it still describes the kernels that run."""
    import hashlib

    h = hashlib.sha256()
    for f in ("topk_impl.cuh", "order_core.cuh", "sel_internal.h", "ptx.cuh", "gather.cu"):
        with open(os.path.join(ROOT, "gather_radix_select_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def stored_traffic(workload: str, kernel: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, one ncu capture) of `kernel`
    on `workload` from the tab-separated table TRAFFIC_FILE (workload, kernel, bytes, source hash), or
    None when absent or taken on other kernel source."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    src = kernel_source_hash()
    for ln in lines:
        cells = ln.split("\t")
        if len(cells) >= 4 and cells[0] == workload and cells[1] == kernel and cells[3].strip() == src:
            try:
                return int(cells[2])
            except ValueError:
                return None
    return None


def cpu_model() -> str:
    """The host CPU's model name (as the kernel reports it), or "" when it cannot be read."""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                k, _, v = ln.partition(":")
                if k.strip().lower() in ("model name", "cpu model") and v.strip():
                    return v.strip()
    except OSError:
        pass
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            k, _, v = ln.partition(":")
            if k.strip() == "Model name" and v.strip():
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return ""


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def shard_plan(w, rank: int, world: int):
    """This rank's share of `world` copies of workload w laid end to end along rows (weak scaling):
    rows partitioned with gather_radix_select_gb300.shard (dual chunks when rows have ends, blocks
    otherwise).  Returns (global rows of this rank, pieces), a piece being (local start, local stop,
    first key batch, stop key batch) of one library call; key batches index `world` copies of the
    workload's key.  One rank: the whole workload in one call."""
    from gather_radix_select_gb300 import shard

    R = w["rows"]
    mode = "dual_chunk" if w["row_end"] is not None else "blocks"
    ranges = shard.partition_rows(R * world, world, mode)[rank]
    grows = shard.rows_of(ranges)
    if w.get("key") is not None:
        glob = shard.call_pieces(ranges, w["rows_per_batch"])
    else:
        glob = [(s, e, 0, 0) for s, e in ranges]
    pieces, at = [], 0
    for s, e, b0, b1 in glob:
        pieces.append((at, at + (e - s), b0, b1))
        at += e - s
    return grows, pieces, mode


class Runner:
    """Device-resident inputs/outputs of one rank's share of a workload and the calls that are timed
    (one rank: the whole workload, one call)."""

    def __init__(self, w, dev, sorted_value=False, rank=0, world=1):
        import torch

        import gather_radix_select_gb300 as g

        self.g, self.torch, self.w, self.dev = g, torch, w, dev
        # value-ordered output instead of the workload's own order (a second launch per step)
        self.sorted_value = sorted_value
        self.sorted_index = w["sorted_index"] and not sorted_value
        self.grows, self.pieces, self.mode = shard_plan(w, rank, world)
        local = self.grows % w["rows"]  # the workload row behind each of this rank's rows
        whole = world == 1
        xb = w["x"] if whole else np.ascontiguousarray(w["x"][local])
        if w["dtype"] == "f32":
            self.x = torch.from_numpy(xb.view(np.int32)).view(torch.float32).to(dev)
        else:
            self.x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
        self.x = self.x[:, :w["cols"]]
        self.rows = len(self.grows)
        self.end = None if w["row_end"] is None else torch.from_numpy(
            w["row_end"] if whole else np.ascontiguousarray(w["row_end"][local])).to(dev)
        self.idx_t = torch.int64 if w["idx_dtype"] == "i64" else torch.int32
        self.key = None
        if w.get("key") is not None:
            key = torch.from_numpy(w["key"].view(np.int16)).view(torch.bfloat16).to(dev)
            self.key = key if whole else torch.cat([key] * world)
            self.gout = torch.empty((self.rows, w["n_gather"], w["d"]), dtype=torch.bfloat16, device=dev)
        self.nan = torch.zeros(1, dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # outputs allocated once (rows padded to 16 bytes), so a step is the library calls alone
        k = w["k"]
        ipad = (k + 3) // 4 * 4 if self.idx_t == torch.int32 else (k + 1) // 2 * 2
        self.out_idx = torch.empty((self.rows, ipad), dtype=self.idx_t, device=dev)
        self.out_val = None
        if w["want_values"]:
            vpad = (k + 3) // 4 * 4 if w["dtype"] == "f32" else (k + 7) // 8 * 8
            self.out_val = torch.empty((self.rows, vpad), dtype=self.x.dtype, device=dev)
        # one fused launch per piece; value order adds the ordering launch (which also gathers)
        per = 1 if not sorted_value else 2
        self.launches_per_step = per * len(self.pieces)

    def local_workload(self):
        """The workload's rows of this rank (for byte counts)."""
        return self.w if len(self.grows) == self.w["rows"] and (self.grows == np.arange(self.rows)).all() \
            else syn.row_subset(self.w, self.grows % self.w["rows"])

    def step(self):
        w = self.w
        for lo, hi, b0, b1 in self.pieces:
            end = None if self.end is None else self.end[lo:hi]
            ov = None if self.out_val is None else self.out_val[lo:hi]
            if self.key is not None:
                self.g.topk_gather(self.x[lo:hi], w["k"], self.key[b0:b1], w["n_gather"], end=end,
                                   sorted_index=self.sorted_index, sorted_value=self.sorted_value,
                                   indices_type=self.idx_t,
                                   return_value=w["want_values"], gather_out=self.gout[lo:hi],
                                   output_idx=self.out_idx[lo:hi], output_val=ov,
                                   nan_flag=self.nan, err_flag=self.err)
            else:
                self.g.topk(self.x[lo:hi], w["k"], end=end, sorted_index=self.sorted_index,
                            sorted_value=self.sorted_value, indices_type=self.idx_t,
                            return_value=w["want_values"], output_idx=self.out_idx[lo:hi], output_val=ov,
                            nan_flag=self.nan, err_flag=self.err)


def time_steps(runner, steps, warmup, flush):
    """Per-step CUDA-event times (ms) with an untimed L2 flush before each step.  flush None: warm
    L2 (the previous step's data may still be cached); a ~0.1 ms GPU sleep (a fixed clock count)
    stands in for the flush so that the host queues the step meanwhile and the events time the step
    alone, not the host's launch latency.  With a flush, one GPU sleep before the first step gives
    the host the same head start."""
    torch = runner.torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        runner.step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if flush is not None:
        # the GPU sleeps (a fixed clock count, ~0.1 ms a step) while the host queues the steps, so no
        # step's events time the host's launch latency (after the synchronize above the first step's
        # flush would otherwise finish before the host has issued its call)
        torch.cuda._sleep(200_000 * steps)
    for a, b in evs:
        if flush is not None:
            flush.zero_()
        else:
            torch.cuda._sleep(200_000)
        a.record(stream)
        runner.step()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def e2e_pieces(w, chunks: int):
    """Row pieces of the end-to-end pipeline: `chunks` blocks of rows, cut where a fused call needs it
    (one key batch per piece unless the piece holds whole batches).  (start, stop, first key batch,
    stop key batch)."""
    from gather_radix_select_gb300 import shard

    blocks = [r for rs in shard.partition_rows(w["rows"], chunks, "blocks") for r in rs]
    if w.get("key") is None:
        return [(s, e, 0, 0) for s, e in blocks]
    return [p for b in blocks for p in shard.call_pieces([b], w["rows_per_batch"])]


def e2e_measure(w, dev, steps, warmup, chunks=4):
    """The step through the public API with host buffers, every copy inside the timed region: the
    inputs go host -> device in row chunks from pinned memory on one stream, each chunk's call runs
    on a second stream as soon as its rows have landed, and its outputs go back to pinned host
    memory on a third, so the copy of chunk j+1, the call on chunk j and the copy back of chunk
    j-1 overlap.  Returns (ms per step, host->device bytes, device->host bytes)."""
    import torch

    import gather_radix_select_gb300 as g

    tdt = torch.float32 if w["dtype"] == "f32" else torch.bfloat16
    host_x = torch.from_numpy(w["x"].view(np.int32 if w["dtype"] == "f32" else np.int16)).view(tdt).pin_memory()
    host_end = None if w["row_end"] is None else torch.from_numpy(w["row_end"]).pin_memory()
    host_key = None
    if w.get("key") is not None:
        host_key = torch.from_numpy(w["key"].view(np.int16)).view(torch.bfloat16).pin_memory()
    idx_t = torch.int64 if w["idx_dtype"] == "i64" else torch.int32
    R, k = w["rows"], w["k"]
    x = torch.empty(host_x.shape, dtype=tdt, device=dev)
    end = None if host_end is None else torch.empty(host_end.shape, dtype=torch.int32, device=dev)
    key = None if host_key is None else torch.empty(host_key.shape, dtype=torch.bfloat16, device=dev)
    # outputs: device buffers written by the calls, pinned host buffers they are read back into
    ipad = (k + 3) // 4 * 4 if idx_t == torch.int32 else (k + 1) // 2 * 2
    out_idx = torch.empty((R, ipad), dtype=idx_t, device=dev)
    out_val = None
    if w["want_values"]:
        vpad = (k + 3) // 4 * 4 if w["dtype"] == "f32" else (k + 7) // 8 * 8
        out_val = torch.empty((R, vpad), dtype=tdt, device=dev)
    gout = None if key is None else torch.empty((R, w["n_gather"], w["d"]), dtype=torch.bfloat16, device=dev)
    h_idx = torch.empty((R, k), dtype=idx_t, pin_memory=True)
    h_val = None if out_val is None else torch.empty((R, k), dtype=tdt, pin_memory=True)
    h_g = None if gout is None else torch.empty(tuple(gout.shape), dtype=torch.bfloat16, pin_memory=True)
    pieces = e2e_pieces(w, chunks)
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)
    h2d = host_x.numel() * host_x.element_size() + (0 if host_end is None else host_end.numel() * 4) + \
        (0 if host_key is None else host_key.numel() * 2)
    d2h = h_idx.numel() * h_idx.element_size() + (0 if h_val is None else h_val.numel() * h_val.element_size()) + \
        (0 if h_g is None else h_g.numel() * 2)

    def one():
        start = torch.cuda.Event()
        start.record(main)
        for st in (s_in, s_run, s_out):
            st.wait_event(start)
        with torch.cuda.stream(s_in):
            if key is not None:
                key.copy_(host_key, non_blocking=True)
        for lo, hi, b0, b1 in pieces:
            landed, done = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                x[lo:hi].copy_(host_x[lo:hi], non_blocking=True)
                if end is not None:
                    end[lo:hi].copy_(host_end[lo:hi], non_blocking=True)
                landed.record(s_in)
            s_run.wait_event(landed)
            xv = x[lo:hi, :w["cols"]]
            ev = None if end is None else end[lo:hi]
            ov = None if out_val is None else out_val[lo:hi]
            if key is not None:
                g.topk_gather(xv, k, key[b0:b1], w["n_gather"], end=ev, sorted_index=w["sorted_index"],
                              indices_type=idx_t, return_value=w["want_values"], output_idx=out_idx[lo:hi],
                              output_val=ov, gather_out=gout[lo:hi], stream=s_run)
            else:
                g.topk(xv, k, end=ev, sorted_index=w["sorted_index"], indices_type=idx_t,
                       return_value=w["want_values"], output_idx=out_idx[lo:hi], output_val=ov, stream=s_run)
            done.record(s_run)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                h_idx[lo:hi].copy_(out_idx[lo:hi, :k], non_blocking=True)
                if h_val is not None:
                    h_val[lo:hi].copy_(out_val[lo:hi, :k], non_blocking=True)
                if h_g is not None:
                    h_g[lo:hi].copy_(gout[lo:hi], non_blocking=True)
        for st in (s_in, s_run, s_out):
            main.wait_stream(st)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    for _ in range(steps):
        one()
    b.record(main)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


def combine_ranks(ms_step: float, nbytes: int, dist, device):
    """Every rank times its own share.  The step time is the slowest rank's; the value is the bytes all
    ranks processed (each rank's own count, summed) per second (GB/s).  dist None = one rank."""
    import torch

    ms_max, total = ms_step, float(nbytes)
    if dist is not None:
        t = torch.tensor([ms_step], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
        b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
        dist.all_reduce(b, op=dist.ReduceOp.SUM)
        total = float(b.item())
    return ms_max, total / (ms_max * 1e-3) / 1e9


def gpu_arm(args):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = syn.workload(args.workload, rows=args.rows)
    if args.topk_only:
        w["key"] = None
    runner = Runner(w, dev, sorted_value=args.sorted_value, rank=rank, world=world)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    peak, peak_kind = measured_peaks()

    # the timed region: K steps, barrier + synchronize on both sides, clocks sampled meanwhile
    for _ in range(args.warmup):
        flush.zero_()
        runner.step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.perf_counter()
    times = time_steps(runner, args.steps, 0, flush)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    if dist:
        dist.barrier()
    ms_step = sum(times) / len(times)
    nbytes = step_bytes(runner.local_workload())  # this rank's rows
    ms_max, value = combine_ranks(ms_step, nbytes, dist, dev)
    nbytes = step_bytes(w)  # per workload copy (one GPU's share)
    err_flag = int(runner.err.item())

    result = None
    if rank == 0 and args.profile:
        result = {"profile_run": True, "workload": args.workload, "sorted_value": args.sorted_value,
                  "ms_per_step": round(ms_max, 5),
                  "value": round(value, 2), "unit": "GB/s", "steps": args.steps, "warmup": args.warmup}
    elif rank == 0:
        kernel_ms = sum(times) / len(times)  # the launch's average duration over the timed region
        achieved = nbytes / (kernel_ms * 1e-3) / 1e9
        e2e_ms, h2d, d2h = e2e_measure(w, dev, max(2, min(args.steps, 10)), 2)
        per = per_workload(args, dev, flush, peak) if not args.no_per_workload else None
        pair = pair_gather_measure(dev, flush, peak) if not args.no_per_workload else None
        blocks = block_measure(dev, flush, peak) if not args.no_per_workload else None
        cpu = cpu_baseline(args.workload)
        import gather_radix_select_gb300 as g

        fused = w.get("key") is not None
        kname = g.kernel_name(runner.x.dtype, w["rows"], w["cols"], w["k"], w["n_gather"] if fused else 0)
        traffic = stored_traffic(args.workload, kname)
        result = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_max, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": w["dtype"],
            "data": "synthetic (seeded; shapes of the workload, no dataset)",
            "config": {"workload": args.workload, "description": w["description"], "rows": w["rows"],
                       "cols": w["cols"], "k": w["k"], "algorithmic_bytes_per_step": nbytes,
                       "rows_per_s": round(w["rows"] * world / (ms_max * 1e-3), 1),
                       "l2": "flushed before every timed step (256 MiB write, untimed)",
                       "parallelism": ("rows of %d workload copies sharded over %d GPUs (%s)" % (world, world, runner.mode))
                       if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                         "kernel": kname + ("<%s,gather>" % w["dtype"] if fused else "<%s>" % w["dtype"]),
                         "algorithmic_bytes": nbytes, "peak_kind": peak_kind},
            "e2e": {"value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 4),
                    "pipeline": "inputs copied in, selected and copied out in 4 row chunks on three streams"},
            "gpu_launches": args.steps * runner.launches_per_step,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "wall_s_timed_region": round(wall, 4),
            "device_err_flag": err_flag,
            "per_workload": per,
            "pair_gather": pair,
            "block_candidates": blocks,
        }
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result


def per_workload(args, dev, flush, peak):
    """Every named workload, a few L2-flushed reps each (median)."""
    import torch

    out = {}
    for name in syn.WORKLOADS:
        w = syn.workload(name)
        r = Runner(w, dev)
        times = time_steps(r, 10, 3, flush)
        ms = statistics.median(times)
        nb = step_bytes(w)
        tb = topk_bytes(w)
        fused = w.get("key") is not None
        warm = statistics.median(time_steps(r, 10, 3, None))
        out[name] = {"kernel": r.g.kernel_name(r.x.dtype, w["rows"], w["cols"], w["k"], w["n_gather"] if fused else 0),
                     "ms": round(ms, 5), "warm_l2_ms": round(warm, 5), "rows_per_s": round(w["rows"] / (ms * 1e-3), 1),
                     "gbs": round(nb / (ms * 1e-3) / 1e9, 2), "frac_of_peak": round(nb / (ms * 1e-3) / 1e9 / peak, 4),
                     "frac_of_nominal": round(nb / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
                     "bytes": nb, "topk_bytes": tb, "fused_gather": w.get("key") is not None}
        t2 = ms
        if w.get("key") is not None:
            # the top-k alone on the same workload (the step above adds the fused gather's bytes)
            w2 = dict(w)
            w2["key"] = None
            r2 = Runner(w2, dev)
            t2 = statistics.median(time_steps(r2, 10, 3, flush))
            out[name]["topk_only_kernel"] = r2.g.kernel_name(r2.x.dtype, w["rows"], w["cols"], w["k"], 0)
            del r2
        out[name]["topk_only_ms"] = round(t2, 5)
        out[name]["topk_only_gbs"] = round(tb / (t2 * 1e-3) / 1e9, 2)
        out[name]["topk_only_frac"] = round(tb / (t2 * 1e-3) / 1e9 / peak, 4)
        # the same step with value-ordered output (selection + ordering launch; same algorithmic bytes)
        r3 = Runner(w, dev, sorted_value=True)
        t3 = statistics.median(time_steps(r3, 10, 3, flush))
        out[name]["value_order_ms"] = round(t3, 5)
        out[name]["value_order_gbs"] = round(nb / (t3 * 1e-3) / 1e9, 2)
        del r3
        del r
        torch.cuda.empty_cache()
    return out


class _Call:
    """A timed call for time_steps."""

    def __init__(self, fn):
        import torch

        self.torch, self.step = torch, fn


def profile_extra(args):
    """--profile-extra pair|block: only the warm-up and timed calls of the double gather or the
    block-level candidate chain (a short run for ncu); prints their median time."""
    import torch

    import gather_radix_select_gb300 as g

    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    if args.profile_extra == "pair":
        w = syn.kl_pair_gather()
        key = torch.from_numpy(w["key"].view(np.int16)).view(torch.bfloat16).to(dev)
        key2 = torch.from_numpy(w["key2"].view(np.int16)).view(torch.bfloat16).to(dev)
        pos = torch.from_numpy(w["pos"]).to(dev)
        out = torch.empty((w["rows"], w["n"], w["d"]), dtype=torch.bfloat16, device=dev)
        out2 = torch.empty((w["rows"], w["n"], w["d2"]), dtype=torch.bfloat16, device=dev)
        call = _Call(lambda: g.gather_rows_pair(key, key2, pos, out=out, out2=out2))
    else:
        w = syn.block_candidates_workload()
        scores = torch.from_numpy(w["scores"].view(np.int16)).view(torch.bfloat16).to(dev)
        key = torch.from_numpy(w["key"].view(np.int16)).view(torch.bfloat16).to(dev)
        pe = torch.from_numpy(w["pos_end"]).to(dev)
        npos = w["topk_blocks"] * w["block_size"]
        pos = torch.empty((w["rows"], npos), dtype=torch.int32, device=dev)
        out = torch.empty((w["rows"], npos, w["d"]), dtype=torch.bfloat16, device=dev)
        call = _Call(lambda: g.block_topk_gather(scores, w["topk_blocks"], w["block_size"], pos_end=pe, key=key,
                                                 out_pos=pos, gather_out=out))
    times = time_steps(call, args.steps, args.warmup, flush)
    return {"profile_run": True, "extra": args.profile_extra, "ms": round(statistics.median(times), 5),
            "steps": args.steps, "warmup": args.warmup}


def pair_gather_measure(dev, flush, peak):
    """The Indexer KL loss's double gather (1024 rows x 512 positions; index key d=128 and
    attention key d=512, compressed length 2048) in one launch, beside the same two gathers
    as separate launches."""
    import torch

    import gather_radix_select_gb300 as g

    w = syn.kl_pair_gather()
    key = torch.from_numpy(w["key"].view(np.int16)).view(torch.bfloat16).to(dev)
    key2 = torch.from_numpy(w["key2"].view(np.int16)).view(torch.bfloat16).to(dev)
    pos = torch.from_numpy(w["pos"]).to(dev)
    R, n, d, d2 = w["rows"], w["n"], w["d"], w["d2"]
    out = torch.empty((R, n, d), dtype=torch.bfloat16, device=dev)
    out2 = torch.empty((R, n, d2), dtype=torch.bfloat16, device=dev)
    uniq = len(np.unique(np.maximum(w["pos"], 0)))
    nbytes = R * n * 4 + uniq * (d + d2) * 2 + R * n * (d + d2) * 2
    t1 = statistics.median(time_steps(_Call(lambda: g.gather_rows_pair(key, key2, pos, out=out, out2=out2)),
                                      10, 3, flush))

    def two():
        g.gather_rows(key, pos, out=out)
        g.gather_rows(key2, pos, out=out2)

    t2 = statistics.median(time_steps(_Call(two), 10, 3, flush))
    res = {"workload": "kl_pair_gather_bf16_1024x512_d128_d512", "ms": round(t1, 5),
           "gbs": round(nbytes / (t1 * 1e-3) / 1e9, 2), "frac_of_peak": round(nbytes / (t1 * 1e-3) / 1e9 / peak, 4),
           "bytes": nbytes, "two_launches_ms": round(t2, 5)}
    del out, out2
    torch.cuda.empty_cache()
    return res


def block_measure(dev, flush, peak):
    """The block-level candidate chain: 1024 rows of 32 block scores (blocks of 64 over
    compressed length 2048), 16 blocks -> 1024 positions a row, causal ends, and the gather
    of the 128-wide key rows at those positions (one launch)."""
    import torch

    import gather_radix_select_gb300 as g

    w = syn.block_candidates_workload()
    scores = torch.from_numpy(w["scores"].view(np.int16)).view(torch.bfloat16).to(dev)
    key = torch.from_numpy(w["key"].view(np.int16)).view(torch.bfloat16).to(dev)
    pe = torch.from_numpy(w["pos_end"]).to(dev)
    R, tb, bs, d = w["rows"], w["topk_blocks"], w["block_size"], w["d"]
    npos = tb * bs
    pos = torch.empty((R, npos), dtype=torch.int32, device=dev)
    out = torch.empty((R, npos, d), dtype=torch.bfloat16, device=dev)
    t = statistics.median(time_steps(_Call(lambda: g.block_topk_gather(scores, tb, bs, pos_end=pe, key=key,
                                                                      out_pos=pos, gather_out=out)), 10, 3, flush))
    # algorithmic bytes: block scores + positions + the key rows at least once + the gathered rows
    nbytes = R * w["n_blocks"] * 2 + R * npos * 4 + w["comp_len"] * d * 2 + R * npos * d * 2
    res = {"workload": "block_candidates_bf16_1024x32_top16x64_gather_d128", "ms": round(t, 5),
           "gbs": round(nbytes / (t * 1e-3) / 1e9, 2), "frac_of_peak": round(nbytes / (t * 1e-3) / 1e9 / peak, 4),
           "bytes": nbytes, "launches": 1}
    del out, pos
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------
# CPU arm: the oracle as it stands, on a bounded sample
# ----------------------------------------------------------------------------

def oracle_step(w, rows_sel):
    import oracle

    s = syn.row_subset(w, rows_sel)
    t0 = time.perf_counter()
    idx, _, _ = oracle.topk(s["x"], w["dtype"], w["k"], row_end=s["row_end"], sorted_index=w["sorted_index"],
                            cols=w["cols"])
    if w.get("key") is not None:
        # gather of the sampled rows, batch by batch (the oracle's own batch rule per block)
        rpb = w["rows_per_batch"]
        for bb in range(w["b"]):
            m = (rows_sel // rpb) == bb
            if m.any():
                oracle.gather_rows(np.ascontiguousarray(w["key"][bb:bb + 1]), idx[m][:, :w["n_gather"]], 1)
    return time.perf_counter() - t0


def oracle_step_parallel(w, rows_sel, workers):
    """oracle_step over the rows split into `workers` chunks on as many threads (the C oracle
    runs without the interpreter lock)."""
    import concurrent.futures

    chunks = [c for c in np.array_split(rows_sel, workers) if len(c)]
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        list(ex.map(lambda c: oracle_step(w, c), chunks))
    return time.perf_counter() - t0


def sample_bytes(w, rows_sel):
    s = syn.row_subset(w, rows_sel)
    s["key"] = w.get("key")
    if s["key"] is not None:
        s["b"], s["comp_len"], s["d"], s["n_gather"] = w["b"], w["comp_len"], w["d"], w["n_gather"]
    return topk_bytes(s) + (gather_bytes(s, fused=True) if s["key"] is not None else 0)


def cpu_baseline(name, budget_s=10.0):
    w = syn.workload(name)
    R = w["rows"]
    # start with a small sample, grow until one pass takes >= ~1 s, then repeat within the budget
    n = min(R, 64)
    while True:
        rows_sel = np.linspace(0, R - 1, n).astype(np.int64)
        dt = oracle_step(w, rows_sel)
        if dt >= 1.0 or n >= R:
            break
        n = min(R, n * 4)
    total, reps = dt, 1
    while total < budget_s and reps < 20:
        total += oracle_step(w, rows_sel)
        reps += 1
    per = total / reps
    nb = sample_bytes(w, rows_sel)
    # the same sample row-parallel over the host's cores (one thread per core, rows split evenly)
    workers = max(1, os.cpu_count() or 1)
    ptimes = [oracle_step_parallel(w, rows_sel, workers) for _ in range(3)]
    pper = statistics.median(ptimes)
    return {"value": round(nb / per / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": "%d of %d rows (evenly spaced), %d passes, %.2f s per pass; single-threaded C full sort "
                      "per row%s" % (len(rows_sel), R, reps, per, " + triple-loop gather" if w.get("key") is not None
                                     else ""),
            "rows_per_s": round(len(rows_sel) / per, 1),
            "row_parallel": {"value": round(nb / pper / 1e9, 4), "unit": "GB/s", "cores": workers,
                             "rows_per_s": round(len(rows_sel) / pper, 1),
                             "sample": "the same rows split over %d threads, median of 3 passes" % workers}}


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    w = syn.workload(args.workload)
    R = w["rows"]
    # each step: a bounded sample of the workload's rows on the oracle
    n = min(R, 64)
    while True:
        rows_sel = np.linspace(0, R - 1, n).astype(np.int64)
        dt = oracle_step(w, rows_sel)
        if dt >= 0.5 or n >= R:
            break
        n = min(R, n * 4)
    for _ in range(args.warmup):
        oracle_step(w, rows_sel)
    times = [oracle_step(w, rows_sel) for _ in range(args.steps)]
    per = sum(times) / len(times)
    nb = sample_bytes(w, rows_sel)
    value = nb / per / 1e9
    sample = "%d of %d rows per step (evenly spaced); single-threaded C full sort per row" % (len(rows_sel), R)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "rows": w["rows"], "cols": w["cols"], "k": w["k"]},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(syn.WORKLOADS))
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="only the warm-up and timed steps of --workload (a short run for ncu)")
    ap.add_argument("--sorted-value", action="store_true",
                    help="with --profile: the workload's step with value-ordered output")
    ap.add_argument("--profile-extra", choices=["pair", "block"],
                    help="only the double gather or the block-level candidate chain (a short run for ncu)")
    ap.add_argument("--topk-only", action="store_true",
                    help="with --profile: the workload's top-k without its fused gather")
    ap.add_argument("--rows", type=int, default=None,
                    help="with --profile: only the workload's first ROWS rows")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if (args.sorted_value or args.topk_only or args.rows is not None) and not args.profile:
        ap.error("--sorted-value, --topk-only and --rows are profiling modes; they need --profile")
    if args.profile_extra:
        print(json.dumps(profile_extra(args)), flush=True)
        return
    res = reference_arm(args) if args.impl == "reference" else gpu_arm(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
