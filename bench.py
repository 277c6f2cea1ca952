"""Benchmark of the indexer top-k + page-table transform on GB300.

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]``

One step is one pass of the whole path over one batch: the plan kernel and
the select + transform kernels (``topk_plan`` + ``topk_transform``).  The
headline workload is throughput: batch 2048 x seq_len 65536 fp32 scores
(q.k dot products), k=512, page size 64, permuted page table (512 MiB of
scores, more than 1.5 times the L2, so not flushed between timed steps;
smaller inputs get a 256 MiB write before every timed step): the shape
the pages quote their bandwidth figures on.  ``value`` is HBM GB/s over the
algorithmic bytes (scores read + seq_lens read + indices written, the page
table excluded as in SGLang PR #26788), timed with CUDA events on the
launching stream.  Secondary entries time the decode (8192 x 8192),
long-context (1/8/32 x 1M, k=2048) and ragged workloads.

``--impl reference`` times the CPU oracle (full sort per row, all host cores)
on a bounded sample of the same workload.  Under torchrun every rank runs the
same per-GPU workload (weak scaling: rows are independent, no collective on
the data path); rank 0 prints the line.  ``--quick`` leaves out the
end-to-end and CPU-baseline legs (for profiler runs); the timed region is the
same.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_indexer_uint32_gb300 import workloads  # noqa: E402

METRIC = "top-k+page-transform HBM GB/s (fraction of peak); µs/call at batch 1, seq 1M"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 7900.0  # GB300 HBM3e nominal; `frac` is against the measured copy bandwidth, `frac_of_spec` this
L2_FLUSH_BYTES = 256 << 20
# The pages' own figures for a workload of the same shape (another machine:
# context for vs_baseline, not a target), in GB/s.
PAGES_GBS = {
    "throughput": (3250.0, "SGLang PR #26788, streaming bandwidth ~3.2-3.3 TB/s at bs >= 2048, seq 65536, "
                           "k=512 (B200); midpoint"),
    "decode": (1563.0, "SGLang PR #26788, decode bucket 1563 GB/s at b=8192, s=8192, k=512 (B200)"),
}


def log(*a):
    print(f"[bench {time.strftime('%H:%M:%S')}]", *a, file=sys.stderr, flush=True)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest() -> str:
    """Digest of the CUDA sources' code (comments and blank space left out, so
    that a comment edit keeps a profile valid)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_indexer_uint32_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = " ".join(text.split())
        h.update(name.encode() + text.encode())
    return h.hexdigest()[:16]


def _profile_summary(workload_name: str):
    """The committed ncu summary of the workload's select kernel, if it was
    taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"select_kernel_{workload_name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m_sha or m_sha.group(1) != source_digest():
        return None
    return text


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch of the select kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    text = _profile_summary(workload_name)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text) if text else None
    return int(m_tr.group(1)) if m_tr else None


def profiled_kernel(workload_name: str) -> str:
    """The select kernel the dispatch launches for the workload, as the
    committed ncu summary names it (its title), when that summary is current."""
    text = _profile_summary(workload_name)
    m = re.match(r"#\s*`([^`]+)`", text) if text else None
    name = m.group(1) if m else "the select kernel(s) of topk_transform"
    return f"{name}; events around the topk_transform call"


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons during the
    timed region: through NVML every 0.2 ms when libnvidia-ml can be loaded
    (reads only), else through nvidia-smi every 200 ms."""

    # NVML clocks-event reason bits (nvml.h) reported by name
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.sm = []
        self.sm_max = []
        self.reasons = set()
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._dev = None
        try:
            import ctypes

            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() == 0:
                dev = ctypes.c_void_p()
                if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(dev)) == 0:
                    self._nvml, self._dev = lib, dev
        except Exception:
            self._nvml = None

    def _nvml_sample(self):
        import ctypes

        mhz, mx, r = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        lib, dev = self._nvml, self._dev
        if lib.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(mhz)) == 0:  # 1 = NVML_CLOCK_SM
            self.sm.append(float(mhz.value))
        if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:
            self.sm_max.append(float(mx.value))
        if lib.nvmlDeviceGetCurrentClocksThrottleReasons(dev, ctypes.byref(r)) == 0:
            for bit, name in self.REASONS.items():
                if r.value & bit:
                    self.reasons.add(name)

    def _smi_sample(self):
        out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.SMI_FIELDS}",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
        if out.returncode != 0 or not out.stdout.strip():
            return
        f = [x.strip() for x in out.stdout.strip().split(",")]
        if f[0].replace(".", "").isdigit():
            self.sm.append(float(f[0]))
        if f[1].replace(".", "").isdigit():
            self.sm_max.append(float(f[1]))
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for i, name in enumerate(names):
            if len(f) > 4 + i and f[4 + i] == "Active":
                self.reasons.add(name)

    def sample_now(self):
        """One sample from the calling thread (the host enqueues a whole timed
        loop in well under its GPU time, so samples taken right after the
        enqueue fall inside the timed region)."""
        try:
            self._nvml_sample() if self._nvml else self._smi_sample()
        except Exception:
            pass

    def _run(self):
        period = 0.0002 if self._nvml else 0.2
        while not self._stop.is_set():
            try:
                self._nvml_sample() if self._nvml else self._smi_sample()
            except Exception:
                pass
            self._stop.wait(period)

    def __enter__(self):
        self.source = "nvml, 0.2 ms" if self._nvml else "nvidia-smi, 200 ms"
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=10)

    def summary(self):
        if not self.sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "source": self.source}
        return {"sm_mhz": statistics.median(self.sm), "sm_max_mhz": max(self.sm_max) if self.sm_max else None,
                "reasons": sorted(self.reasons), "samples": len(self.sm), "source": self.source}


def build_workload(name: str, shard: int = 0) -> workloads.Workload:
    """The named workload; shard r (rank r of a multi-GPU run) draws its own
    batch of the same shape from its own seed."""
    if name == "decode":
        return workloads.decode(shard=shard)
    if name == "throughput":
        return workloads.throughput(shard=shard)
    if name.startswith("long"):
        return workloads.long_context(int(name[4:] or 1), shard=shard)
    if name == "ragged":
        return workloads.ragged(shard=shard)
    if name == "tiny":
        return workloads.tiny()
    raise ValueError(name)


def config_of(wl: workloads.Workload, name: str, world: int) -> dict:
    eff = np.clip(wl.seq_lens.astype(np.int64), 0, wl.max_seq_len)
    return {"workload": wl.name, "kind": name, "batch": wl.batch, "seq_len": int(eff.max()),
            "sum_seq_len": int(eff.sum()), "k": wl.k, "page_size": wl.page_size, "row_stride": wl.row_stride,
            "raw_output": wl.want_raw, "global_batch": wl.batch * world, "parallelism": f"dp{world}",
            "sharding": "each rank selects its own batch of this shape; no collective on the data path",
            "launch": "plan and transform replayed from CUDA graphs; events on the launching stream"}


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest value of x over all ranks (x itself on one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: int, world: int, steps: int, total_ms_max: float) -> float:
    """Whole-job throughput: the bytes all ranks processed over the slowest
    rank's time for the timed steps."""
    return bytes_per_rank_step * world * steps / (total_ms_max / 1e3) / 1e9


def l2_policy(scores_bytes: int, l2_bytes: int) -> tuple:
    """(flush?, description).  Scores of at least 1.5 times the L2 size are
    not flushed between timed steps: each step streams them through L2 in the
    same order, so a step's reads have replaced what the previous step left
    there before they come back to it.  Smaller inputs get a write of
    L2_FLUSH_BYTES before every timed step."""
    if 2 * scores_bytes >= 3 * l2_bytes:
        return False, (f"not flushed: the scores ({scores_bytes / 2**20:.0f} MiB) are more than 1.5 times the "
                       f"{l2_bytes / 2**20:.0f} MiB L2")
    return True, f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)"


def time_gpu(wl, steps: int, warmup: int, local: int, world: int, want_clocks: bool):
    import torch
    import torch.distributed as dist

    from sparse_attention_indexer_uint32_gb300 import _lib, api

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    do_flush, l2_desc = l2_policy(int(wl.scores.nbytes), int(torch.cuda.get_device_properties(dev).L2_cache_size))
    stream = torch.cuda.current_stream(dev)
    scores = torch.from_numpy(wl.scores).to(dev)
    seq = torch.from_numpy(wl.seq_lens).to(dev)
    table = torch.from_numpy(wl.page_table).to(dev)
    out = torch.empty((wl.batch, wl.k), dtype=torch.int32, device=dev)
    raw = torch.empty((wl.batch, wl.k), dtype=torch.int32, device=dev) if wl.want_raw else None
    ws = torch.zeros(_lib.topk_plan_workspace_bytes(wl.batch), dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        if do_flush:
            flush_buf.fill_(1.0)

    def step():
        _lib.topk_plan(seq, wl.batch, wl.max_seq_len, ws, stream)
        _lib.topk_transform(scores, wl.row_stride, seq, wl.batch, wl.max_seq_len, table, wl.page_table.shape[1],
                            wl.page_size, wl.k, out, raw, ws, stream)

    for _ in range(warmup):
        flush_l2()
        step()
    torch.cuda.synchronize(dev)
    # the plan + the select kernel(s) topk_transform enqueues for this shape
    launches_per_step = 1 + _lib.topk_transform_launches(wl.batch, wl.max_seq_len, wl.k)

    # A step (plan + transform) is replayed from one CUDA graph, as a serving
    # loop would run it: host launch latency stays out of the timed region and
    # the transform's programmatic launch overlaps the plan's tail.
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        _lib.topk_plan(seq, wl.batch, wl.max_seq_len, ws)
        _lib.topk_transform(scores, wl.row_stride, seq, wl.batch, wl.max_seq_len, table, wl.page_table.shape[1],
                            wl.page_size, wl.k, out, raw, ws)
    # The same two calls as two graphs, to time the select kernel(s) alone.
    g_plan, g_sel = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plan):
        _lib.topk_plan(seq, wl.batch, wl.max_seq_len, ws)
    with torch.cuda.graph(g_sel):
        _lib.topk_transform(scores, wl.row_stride, seq, wl.batch, wl.max_seq_len, table, wl.page_table.shape[1],
                            wl.page_size, wl.k, out, raw, ws)
    # plan -> transform -> a dependent consumer (the stand-alone page transform
    # of the raw output, launched with programmatic serialization: it may be
    # placed once every select block has written its output and triggered).
    raw_c = torch.empty((wl.batch, wl.k), dtype=torch.int32, device=dev)
    out_c = torch.empty((wl.batch, wl.k), dtype=torch.int32, device=dev)
    g_chain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_chain):
        _lib.topk_plan(seq, wl.batch, wl.max_seq_len, ws)
        _lib.topk_transform(scores, wl.row_stride, seq, wl.batch, wl.max_seq_len, table, wl.page_table.shape[1],
                            wl.page_size, wl.k, out, raw_c, ws)
        _lib.topk_page_transform(raw_c, wl.batch, wl.k, table, wl.page_table.shape[1], wl.page_size, out_c)
    for _ in range(2):
        flush_l2()
        g_step.replay()
        flush_l2()
        g_plan.replay()
        g_sel.replay()
        flush_l2()
        g_chain.replay()
    torch.cuda.synchronize(dev)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ev3 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local) if want_clocks else None
    if sampler:
        sampler.__enter__()
    t_wall = time.perf_counter()
    for e0, e1 in ev:
        flush_l2()
        e0.record(stream)
        g_step.replay()
        e1.record(stream)
    if sampler:
        while not ev[-1][1].query():  # the GPU is still in the timed steps
            sampler.sample_now()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    if sampler:
        sampler.__exit__(None, None, None)
    if world > 1:
        dist.barrier()
    # Split timing (after the timed region): the plan, then the select kernel(s).
    for e0, e1, e2 in ev3:
        flush_l2()
        e0.record(stream)
        g_plan.replay()
        e1.record(stream)
        g_sel.replay()
        e2.record(stream)
    torch.cuda.synchronize(dev)
    evc = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evc:
        flush_l2()
        e0.record(stream)
        g_chain.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    chain_ms = [e0.elapsed_time(e1) for e0, e1 in evc]
    if not (out_c.cpu() == out.cpu()).all():  # the consumer re-derives out from the raw output
        raise AssertionError("the chained consumer's output differs from the transform's own")
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    plan_ms = [e0.elapsed_time(e1) for e0, e1, _ in ev3]
    sel_ms = [e1.elapsed_time(e2) for _, e1, e2 in ev3]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    flags = _lib.topk_read_flags(ws)
    res = {"total_ms": total_ms, "step_ms": step_ms, "plan_ms": plan_ms, "select_ms": sel_ms, "chain_ms": chain_ms,
           "wall_s": t_wall, "flags": flags, "launches_per_step": launches_per_step,
           "clocks": sampler.summary() if sampler else None, "out": out.cpu().numpy(), "l2": l2_desc}
    del scores, flush_buf
    return res


def time_e2e(wl, steps: int, warmup: int, local: int, chunks: int = 4, copy_streams: int = 1):
    """Same metric through the public API from pinned host buffers: every step
    copies the step's inputs host->device, plans and transforms, and copies the
    result device->host.  The batch is cut into `chunks` row ranges; each
    range's inputs go up on one of `copy_streams` copy streams, and its plan +
    transform + result copy run on the compute stream as soon as that range
    has landed, so copies and selection overlap.  Consecutive steps overlap as
    a serving loop's would: a range's next copy waits only until this step's
    selection of that range is done with the device buffer.  (On GB300 the
    host->device copy runs near 200 GB/s whatever the number of copy streams,
    so the step is copy-bound; 4 ranges on one copy stream measured best.)"""
    import torch

    from sparse_attention_indexer_uint32_gb300 import _lib

    dev = torch.device("cuda", local)
    comp = torch.cuda.current_stream(dev)
    cstreams = [torch.cuda.Stream(dev) for _ in range(copy_streams)]
    h_scores = torch.from_numpy(wl.scores).pin_memory()
    h_seq = torch.from_numpy(wl.seq_lens).pin_memory()
    h_table = torch.from_numpy(wl.page_table).pin_memory()
    h_out = torch.empty((wl.batch, wl.k), dtype=torch.int32).pin_memory()
    d_scores = torch.empty_like(h_scores, device=dev)
    d_seq = torch.empty_like(h_seq, device=dev)
    d_table = torch.empty_like(h_table, device=dev)
    d_out = torch.empty((wl.batch, wl.k), dtype=torch.int32, device=dev)
    cuts = np.linspace(0, wl.batch, min(chunks, wl.batch) + 1).astype(int)
    ranges = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    ws = [torch.zeros(_lib.topk_plan_workspace_bytes(b - a), dtype=torch.uint8, device=dev) for a, b in ranges]
    landed = [torch.cuda.Event() for _ in ranges]
    freed = [torch.cuda.Event() for _ in ranges]

    def step():
        for i, (a, b) in enumerate(ranges):
            cs = cstreams[i % len(cstreams)]
            cs.wait_event(freed[i])  # the previous step's selection of this range is done with its inputs
            with torch.cuda.stream(cs):
                d_scores[a:b].copy_(h_scores[a:b], non_blocking=True)
                d_seq[a:b].copy_(h_seq[a:b], non_blocking=True)
                d_table[a:b].copy_(h_table[a:b], non_blocking=True)
            landed[i].record(cs)
        for i, (a, b) in enumerate(ranges):
            comp.wait_event(landed[i])
            _lib.topk_plan(d_seq[a:b], b - a, wl.max_seq_len, ws[i], comp)
            _lib.topk_transform(d_scores[a:b], wl.row_stride, d_seq[a:b], b - a, wl.max_seq_len, d_table[a:b],
                                wl.page_table.shape[1], wl.page_size, wl.k, d_out[a:b], None, ws[i], comp)
            freed[i].record(comp)
            h_out[a:b].copy_(d_out[a:b], non_blocking=True)

    for i in range(len(ranges)):
        freed[i].record(comp)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for cs in cstreams:  # no copy of the timed steps starts before e0
        cs.wait_event(e0)
    for _ in range(steps):
        step()
    e1.record(comp)  # the compute stream waited for every range's copy
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    h2d = h_scores.numel() * 4 + h_seq.numel() * 4 + h_table.numel() * 4
    d2h = h_out.numel() * 4
    # The bound on this host: the same steps' host->device copies alone (the
    # same ranges on the same copy streams, nothing selected).
    def copies():
        for i, (a, b) in enumerate(ranges):
            with torch.cuda.stream(cstreams[i % len(cstreams)]):
                d_scores[a:b].copy_(h_scores[a:b], non_blocking=True)
                d_seq[a:b].copy_(h_seq[a:b], non_blocking=True)
                d_table[a:b].copy_(h_table[a:b], non_blocking=True)

    copies()
    torch.cuda.synchronize(dev)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(comp)
    for cs in cstreams:
        cs.wait_event(c0)
    for _ in range(steps):
        copies()
    for cs in cstreams:
        comp.wait_stream(cs)
    c1.record(comp)
    torch.cuda.synchronize(dev)
    copy_gbs = steps * h2d / (c0.elapsed_time(c1) * 1e-3) / 1e9
    return ms, h2d, d2h, copy_gbs


def oracle_sample_time(wl, target_s: float = 12.0):
    """Times the oracle (all host cores) on a bounded row sample of the workload."""
    import oracle

    cores = os.cpu_count() or 1
    eff = np.clip(wl.seq_lens.astype(np.int64), 0, wl.max_seq_len)
    # calibrate on a few rows, then size the sample for ~target_s of wall time
    rows = np.arange(min(wl.batch, max(1, cores)))
    t0 = time.perf_counter()
    oracle.topk_transform(wl.scores[rows], wl.seq_lens[rows], wl.page_table[rows], wl.page_size, wl.k,
                          max_seq_len=wl.max_seq_len, want_raw=False, nthreads=cores)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(wl.batch, max(len(rows), len(rows) * target_s / dt)))
    rows = np.arange(n)
    t0 = time.perf_counter()
    oracle.topk_transform(wl.scores[rows], wl.seq_lens[rows], wl.page_table[rows], wl.page_size, wl.k,
                          max_seq_len=wl.max_seq_len, want_raw=False, nthreads=cores)
    dt = time.perf_counter() - t0
    nbytes = int(4 * eff[rows].sum() + 4 * n + 4 * n * wl.k)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {wl.batch} rows of {wl.name}, {dt:.2f} s wall on {cores} threads"}


def check_timed_rows(wl, out, count: int = 64, seed: int = 0) -> dict:
    """Re-checks the output of the timed run on sampled rows, without the
    oracle: positions are recovered through the inverse of the row's page
    table, then each row must hold min(k, L) distinct in-range positions, no
    unselected score above a selected one, and ties at the k-th score taken
    at the smallest positions.  Raises on a failure."""
    rng = np.random.default_rng(seed)
    rows = sorted(set(rng.choice(wl.batch, size=min(count, wl.batch), replace=False).tolist()) | {0, wl.batch - 1})
    P = wl.page_size
    lp = P.bit_length() - 1
    for b in rows:
        L = int(min(max(int(wl.seq_lens[b]), 0), wl.max_seq_len))
        n = min(wl.k, L)
        o = out[b].astype(np.int64)
        if not (o[n:] == -1).all():
            raise AssertionError(f"row {b}: padding is not -1")
        table = wl.page_table[b].astype(np.int64)
        pages = -(-L // P)
        order = np.argsort(table[:pages], kind="stable")
        page_id = (o[:n] & 0xFFFFFFFF) >> lp
        k_pos = np.searchsorted(table[:pages][order], page_id)
        if n and ((k_pos >= pages).any() or (table[:pages][order][np.minimum(k_pos, pages - 1)] != page_id).any()):
            raise AssertionError(f"row {b}: an output is not a page of the row's table")
        raw = order[np.minimum(k_pos, pages - 1)] * P + (o[:n] & (P - 1))
        if n and (len(np.unique(raw)) != n or raw.min() < 0 or raw.max() >= L):
            raise AssertionError(f"row {b}: positions repeat or leave the row")
        if 0 < n < L:
            x = wl.scores[b, :L]
            sel = np.zeros(L, dtype=bool)
            sel[raw] = True
            t = x[sel].min()
            if x[~sel].max() > t:
                raise AssertionError(f"row {b}: an unselected score beats a selected one")
            tied = np.nonzero(x == t)[0]
            if sel[tied].any() and (~sel[tied]).any() and tied[sel[tied]].max() > tied[~sel[tied]].min():
                raise AssertionError(f"row {b}: ties at the k-th score not taken smallest position first")
    return {"rows": len(rows), "result": "ok", "how": "page-table inverse + order properties, no oracle"}


def gpu_line(name: str, steps: int, warmup: int, world: int, rank: int, local: int, full: bool,
             quick: bool = False):
    log("workload", name)
    wl = build_workload(name, shard=rank)
    nbytes = wl.algorithmic_bytes()
    r = time_gpu(wl, steps, warmup, local, world, want_clocks=full)
    log("timed", name, f"{r['total_ms'] / steps:.4f} ms/step", "flags", r["flags"])
    peak, peak_kind = measured_peak()
    ms_step = r["total_ms"] / steps
    sel_avg = statistics.mean(r["select_ms"])
    value = job_gbs(nbytes, world, steps, r["total_ms"])
    achieved = nbytes / (sel_avg / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / PAGES_GBS[name][0], 4) if name in PAGES_GBS else None,
        "vs_baseline_source": PAGES_GBS[name][1] if name in PAGES_GBS else None,
        "dtype": "f32 scores, u32 keys, i32 indices", "data": "synthetic (seeded)",
        "config": {**config_of(wl, name, world), "l2": r["l2"]},
        "us_per_call": round(ms_step * 1e3, 2),
        "step_us_p10_p50_p90": [round(float(np.percentile(r["step_ms"], q)) * 1e3, 2) for q in (10, 50, 90)],
        "timed_output_check": check_timed_rows(wl, r["out"]),
        "plan_us": round(statistics.mean(r["plan_ms"]) * 1e3, 2),
        "select_us": round(sel_avg * 1e3, 2),
        "chain_us": round(statistics.mean(r["chain_ms"]) * 1e3, 2),
        "chain": "plan + transform (raw output too) + a consumer kernel (the stand-alone page transform of the "
                 "raw output) launched with programmatic serialization, one graph, events around it",
        "algorithmic_bytes_per_step": nbytes,
        "gpu_launches": r["launches_per_step"] * steps,
        "device_flags": r["flags"],
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(name),
                     "frac_of_spec": round(achieved / SPEC_HBM_GBS, 4), "spec_peak": SPEC_HBM_GBS,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                     "kernel": profiled_kernel(name)},
    }
    if full and not quick:
        e2e_steps = max(3, min(steps, 10))
        ms, h2d, d2h, copy_gbs = time_e2e(wl, e2e_steps, 2, local)
        log("e2e", f"{ms:.3f} ms/step, the copies alone {copy_gbs:.1f} GB/s")
        import torch

        ms = max_over_ranks(ms, world, torch.device("cuda", local))
        line["e2e"] = {"value": round(job_gbs(nbytes, world, 1, ms), 2), "unit": "GB/s",
                       "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world,
                       "ms_per_step": round(ms, 4),
                       # the same host->device copies alone, on this host: the step's bound
                       # (its rate differs between hosts)
                       "h2d_copy_gbs": round(copy_gbs, 1)}
        if rank == 0 and world == 1:
            line["cpu_baseline"] = oracle_sample_time(wl)
            log("cpu baseline", line["cpu_baseline"])
    if full:
        line["clocks"] = r["clocks"]
    elif rank == 0 and world == 1 and not quick:
        # the oracle beside every workload's GPU figure (a shorter sample)
        line["cpu_baseline"] = oracle_sample_time(wl, target_s=3.0)
    return line


def parse_tuning(spec: str) -> dict:
    """'name=value,...' -> {name: int}, names checked against the library's
    tuning struct (topk_tuning_t in include/topkidx.h)."""
    from sparse_attention_indexer_uint32_gb300 import _lib

    fields = {name for name, _ in _lib.topk_tuning_t._fields_}
    out = {}
    for item in [x.strip() for x in spec.split(",") if x.strip()]:
        name, sep, value = item.partition("=")
        if not sep or name not in fields:
            raise ValueError(f"--tuning: {item!r} is not name=value with a topk_tuning_t field name")
        out[name] = int(value)
    return out


def apply_tuning(kv: dict) -> None:
    from sparse_attention_indexer_uint32_gb300 import _lib

    t = _lib.topk_get_tuning()
    for name, value in kv.items():
        setattr(t, name, value)
    _lib.topk_set_tuning(t)  # the library validates the values


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="throughput",
                    help="headline workload: batch 2048 x 64K, k=512, the shape the bandwidth figures are quoted on")
    ap.add_argument("--secondary", default="decode,long1,long8,long32,ragged",
                    help="comma list of extra workloads timed after the headline one ('' for none)")
    ap.add_argument("--tuning", default="",
                    help="comma list of name=value library tuning knobs set before timing, e.g. warp_rows=1 "
                         "(recorded in each line's config)")
    ap.add_argument("--quick", action="store_true",
                    help="leave out the end-to-end and CPU-baseline legs (profiler runs); the timed region is unchanged")
    args = ap.parse_args()
    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return
        wl = build_workload(args.workload)
        times, last = [], None
        # about two minutes of host work in all, whatever --steps is
        per_step = max(0.5, min(8.0, 120.0 / max(1, args.steps)))
        for _ in range(args.warmup):
            oracle_sample_time(wl, target_s=min(2.0, per_step))
        for _ in range(args.steps):
            last = oracle_sample_time(wl, target_s=per_step)
            times.append(last["value"])
        v = statistics.mean(times)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 scores, i32 indices", "data": "synthetic (seeded)",
            "config": {**config_of(wl, args.workload, 1), "l2": "n/a (host)",
                       "launch": "the CPU oracle on all host threads, one bounded sample per step"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    tuning_kv = parse_tuning(args.tuning)
    if tuning_kv:
        apply_tuning(tuning_kv)
    line = gpu_line(args.workload, args.steps, args.warmup, world, rank, local, full=True, quick=args.quick)
    if tuning_kv:
        line["config"]["tuning"] = tuning_kv
    extra = []
    for name in [s for s in args.secondary.split(",") if s]:
        try:
            sub = gpu_line(name, max(3, args.steps // 2), max(3, args.warmup // 2), world, rank, local, full=False,
                           quick=args.quick)
            extra.append({k: sub[k] for k in ("config", "value", "vs_baseline", "us_per_call", "select_us", "plan_us",
                                              "chain_us", "roofline", "device_flags", "cpu_baseline") if k in sub})
            if tuning_kv:
                extra[-1]["config"]["tuning"] = tuning_kv
        except Exception as e:  # report, never hide
            extra.append({"workload": name, "error": repr(e)})
    line["secondary"] = extra
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
