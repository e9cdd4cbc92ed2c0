#!/usr/bin/env python
"""Benchmark: length-aware GQA decode attention on GB300.

One step = one fd_decode call over the batched ragged workload (8 sequences,
lengths uniform in [1024, 32768] from the seed, capacity 32768, 6-row causal
window, 16 q / 4 kv heads, head_dim 128 x 2 = 256, bf16 cache).  The metric is
KV-read HBM bandwidth: the K and V bytes of the filled prefixes
(sum_b L_b * Hkv * d * 2 bytes * 2 tensors) divided by the step time.  The
filled prefixes (~0.5 GB) are larger than L2, so no flush is needed between
steps.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on the
host cores on a bounded sample of the same workload instead.

Multi-GPU (torchrun, one process per GPU): every rank runs its own replica on
its own batch (no collective on the data path); ``value`` sums the bytes of
all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KV-read HBM GB/s per decode-attention call"
UNIT = "GB/s"
WORKLOAD = "ragged"
WORKLOAD_DESC = ("batched ragged decode: B=8, kv_len uniform[1024,32768] (seed), "
                 "cap=32768, n_q=6 causal, Hq=16, Hkv=4, head_dim=256, bf16 K/V")
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers
def rank_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(x, world, device=None):
    """The largest x over the ranks (the slowest replica's time)."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank, world, ms_max):
    """Whole-job GB/s: every replica's bytes over the slowest replica's time."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kv_bytes(lengths, Hkv, d, esize):
    return sum(int(L) for L in lengths) * Hkv * d * esize * 2


# The sources the headline kernel (the tensor-core kernel over flat caches)
# is built from: its template, its launch unit and the headers they include.
TC_KERNEL_SOURCES = ("fd_device.cuh", "fd_internal.h", "fd_launch.h", "fd_ptx.cuh", "fd_tc.cu",
                     "fd_tc_kernel.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_preallocated_gb300", "csrc")
    for name in TC_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.txt" % workload)
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sources") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- workloads
def append_inputs(name, seed, device):
    """A named workload as one fused append step: its window's rows (n_q per
    sequence) are new, written at L - n_q and attended; the lengths passed are
    L - n_q, and the timed calls leave them there."""
    from decode_attention_preallocated_gb300 import workloads as W
    inp = W.workload(name, seed=seed, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(7)
    B, n, _, d = inp.q.shape
    Hkv = inp.k.shape[1]
    inp.k_new = W.randn_bf16((B, n, Hkv, d), g, device)
    inp.v_new = W.randn_bf16((B, n, Hkv, d), g, device)
    inp.lengths_host = [L - n for L in inp.lengths_host]
    inp.kv_lengths = inp.kv_lengths - n
    return inp


def make_inputs(name, seed, device):
    """A named workload, "append_<workload>" (that workload as one fused
    append step), or "sweep:L,B,Hq,Hkv,d,n_q": B sequences all of length L
    in a cache of capacity L + 1000 (causal when n_q > 1)."""
    from decode_attention_preallocated_gb300 import workloads as W
    if name.startswith("append_"):
        return append_inputs(name[len("append_"):], seed, device)
    if name.startswith("sweep:"):
        L, B, Hq, Hkv, d, nq = (int(x) for x in name[6:].split(","))
        return W.dense_inputs(B, nq, Hq, Hkv, d, L + 1000, [L] * B, seed, nq > 1,
                              device=device, name=name)
    return W.workload(name, seed=seed, device=device)


def workload_desc(name):
    if name == WORKLOAD:
        return WORKLOAD_DESC
    if name.startswith("sweep:"):
        L, B, Hq, Hkv, d, nq = name[6:].split(",")
        return ("uniform decode: B=%s, kv_len=%s, cap=kv_len+1000, n_q=%s%s, Hq=%s, Hkv=%s, "
                "head_dim=%s, bf16 K/V" % (B, L, nq, " causal" if int(nq) > 1 else "", Hq, Hkv, d))
    return name


def call_fn(inp, out, ws, kernel, num_ctas=0):
    from decode_attention_preallocated_gb300 import fd
    if getattr(inp, "k_new", None) is not None:
        # fused append step; the lengths are left as they are, so every timed
        # call appends the same rows at the same positions
        return lambda: fd.decode_append(inp.q, inp.k, inp.v, inp.k_new, inp.v_new,
                                        inp.kv_lengths, causal=inp.causal, scale=inp.scale,
                                        update_lengths=False, out=out, workspace=ws,
                                        kernel=kernel, num_ctas=num_ctas)
    if getattr(inp, "mask", None) is not None:
        return lambda: fd.decode_masked(inp.q, inp.k, inp.v, inp.kv_lengths, inp.mask,
                                        n_q=inp.n_q, causal=inp.causal, scale=inp.scale, out=out,
                                        workspace=ws, kernel=kernel, num_ctas=num_ctas)
    if inp.block_table is not None:
        return lambda: fd.decode_paged(inp.q, inp.k, inp.v, inp.block_table, inp.kv_lengths,
                                       n_q=inp.n_q, causal=inp.causal, scale=inp.scale,
                                       k_scale=inp.k_scale, v_scale=inp.v_scale, out=out,
                                       workspace=ws, kernel=kernel, num_ctas=num_ctas)
    if inp.idx is not None:
        return lambda: fd.decode_gather(inp.q, inp.k, inp.v, inp.idx, scale=inp.scale, out=out,
                                        workspace=ws, kernel=kernel, num_ctas=num_ctas,
                                        bias=getattr(inp, "bias", None), k_scale=inp.k_scale,
                                        v_scale=inp.v_scale)
    if inp.k.dtype == torch.int8:
        return lambda: fd.decode_int8(inp.q, inp.k, inp.v, inp.k_scale, inp.v_scale,
                                      inp.kv_lengths, n_q=inp.n_q, causal=inp.causal,
                                      scale=inp.scale, out=out, workspace=ws, kernel=kernel,
                                      num_ctas=num_ctas)
    return lambda: fd.decode(inp.q, inp.k, inp.v, inp.kv_lengths, n_q=inp.n_q,
                             causal=inp.causal, scale=inp.scale, out=out, workspace=ws,
                             kernel=kernel, num_ctas=num_ctas)


def algorithmic_bytes(inp):
    B, n_q, Hq, d = inp.q.shape
    Hkv = inp.k.shape[1]
    if inp.idx is not None:
        valid = int(((inp.idx >= 0) & (inp.idx < inp.k.shape[2])).sum())
        if inp.k.dtype == torch.int8:   # codes plus the two fp32 scales of each cell
            return valid * Hkv * (d * 2 + 8)
        return valid * Hkv * d * 2 * 2
    es = 1 if inp.k.dtype == torch.int8 else 2
    if getattr(inp, "mask", None) is not None:
        # masked prefix: the K / V rows of the 32-position chunks some query
        # row sees (the granularity at which the scan skips)
        chunks = 0
        for b_, L in enumerate(inp.lengths_host):
            m = inp.mask[b_, :, :L]
            pad = (-L) % 32
            if pad:
                m = torch.nn.functional.pad(m, (0, pad), value=-float("inf"))
            chunks += int((m.reshape(m.shape[0], -1, 32) != -float("inf")).any(2).any(0).sum())
        return chunks * 32 * Hkv * d * 2 * 2
    if getattr(inp, "k_new", None) is not None:
        # fused append: the new rows are read once and written once, and the
        # attention reads the prefix including them
        n = inp.k_new.shape[1]
        return kv_bytes([L + n for L in inp.lengths_host], Hkv, d, 2) + 2 * kv_bytes([n] * B, Hkv, d, 2)
    b = kv_bytes(inp.lengths_host, Hkv, d, es)
    if es == 1:
        b += sum(inp.lengths_host) * Hkv * 4 * 2   # fp32 per-token scales
    return b


def time_calls(fn, n, stream):
    """Average ms per call of n back-to-back calls (CUDA events on `stream`)."""
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / n


GRAPH_CALLS = 50   # decode calls captured per CUDA graph


def capture(fn, calls, stream):
    """A CUDA graph of `calls` back-to-back calls of fn on `stream` (the
    library allocates nothing and reads no device data on the host, so a
    call captures as-is; a decode loop replays its step graph the same way).
    Calls still running on another stream finish first: a workspace serves
    one stream at a time."""
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls):
            fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, calls, replays, stream):
    """Average ms per call over `replays` replays of a `calls`-call graph."""
    g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(replays):
            g.replay()
        b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / (calls * replays)


def time_stats(fn, stream, calls=10, replays=20):
    """Per-call time (us) over `replays` individually timed replays of a
    graph of `calls` back-to-back calls: mean, median, min and p90 of the
    per-replay averages."""
    g = capture(fn, calls, stream)
    g.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for r in range(replays):
            g.replay()
            evs[r + 1].record(stream)
    evs[-1].synchronize()
    per = sorted(1e3 * evs[r].elapsed_time(evs[r + 1]) / calls for r in range(replays))
    del g
    p90 = per[min(len(per) - 1, int(math.ceil(0.9 * len(per))) - 1)]
    return {"mean": sum(per) / len(per), "median": statistics.median(per), "min": per[0],
            "p90": p90}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def workspace_for(inp, device):
    from decode_attention_preallocated_gb300 import fd
    B, n_q, Hq, d = inp.q.shape
    Hkv = inp.k.shape[1]
    g = Hq // Hkv
    if inp.idx is not None:
        return fd.Workspace(B * n_q * Hkv, g, 256, 4096, device=device)
    # int8 caches with more than 32 rows run on the tensor cores in parts of
    # the query heads, a segment each (at most one per query head)
    parts = g if inp.k.dtype == torch.int8 and g * n_q > 32 else 1
    return fd.Workspace(B * Hkv * parts, g * n_q, 256, 4096, device=device)


# ------------------------------------------------------------ CPU oracle
def oracle_sample(inp_cpu, budget_s=10.0, max_calls=50):
    """Time the fp64 oracle on the host cores on whole sequences of the
    workload until ~budget_s of CPU work; returns (GB/s, threads, sample text)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    B = inp_cpu.q.shape[0]
    bytes_done, t_used, seqs = 0, 0.0, 0
    b = 0
    while t_used < budget_s and seqs < max_calls:
        sl = slice(b, b + 1)
        t0 = time.perf_counter()
        oracle_call(inp_cpu, sl)
        t_used += time.perf_counter() - t0
        sub = sub_inputs(inp_cpu, sl)
        bytes_done += algorithmic_bytes(sub)
        seqs += 1
        b = (b + 1) % B
    gbs = bytes_done / t_used / 1e9
    sample = "%d whole sequence(s) of the workload (%.1f MB of KV), %.1f s" % (
        seqs, bytes_done / 1e6, t_used)
    return gbs, cores, sample


def cpu_view(inp):
    from decode_attention_preallocated_gb300 import workloads as W
    return W.DecodeInputs(
        q=inp.q.cpu(), k=inp.k.cpu(), v=inp.v.cpu(), kv_lengths=inp.kv_lengths.cpu(),
        n_q=inp.n_q, causal=inp.causal, scale=inp.scale,
        k_scale=None if inp.k_scale is None else inp.k_scale.cpu(),
        v_scale=None if inp.v_scale is None else inp.v_scale.cpu(),
        idx=None if inp.idx is None else inp.idx.cpu(),
        lengths_host=list(inp.lengths_host), name=inp.name,
        mask=None if getattr(inp, "mask", None) is None else inp.mask.cpu())


def sub_inputs(inp, sl):
    """Sequences `sl` of a workload (CPU view)."""
    cut = lambda t: None if t is None else t[sl]  # noqa: E731
    return type(inp)(q=inp.q[sl], k=inp.k[sl], v=inp.v[sl], kv_lengths=inp.kv_lengths[sl],
                     n_q=inp.n_q, causal=inp.causal, scale=inp.scale, k_scale=cut(inp.k_scale),
                     v_scale=cut(inp.v_scale), idx=cut(inp.idx),
                     lengths_host=inp.lengths_host[sl], mask=cut(getattr(inp, "mask", None)))


def oracle_call(inp_cpu, sl):
    """The fp64 oracle on the sequences `sl` of a workload (CPU view)."""
    import oracle
    if getattr(inp_cpu, "mask", None) is not None:
        return oracle.masked(inp_cpu.q[sl], inp_cpu.k[sl], inp_cpu.v[sl],
                             inp_cpu.lengths_host[sl], inp_cpu.mask[sl], inp_cpu.n_q,
                             inp_cpu.causal, inp_cpu.scale)
    if inp_cpu.idx is not None:
        return oracle.gather(inp_cpu.q[sl], inp_cpu.k[sl], inp_cpu.v[sl], inp_cpu.idx[sl],
                             inp_cpu.scale,
                             None if inp_cpu.k_scale is None else inp_cpu.k_scale[sl],
                             None if inp_cpu.v_scale is None else inp_cpu.v_scale[sl])
    return oracle.dense(inp_cpu.q[sl], inp_cpu.k[sl], inp_cpu.v[sl],
                        inp_cpu.lengths_host[sl], inp_cpu.n_q, inp_cpu.causal, inp_cpu.scale,
                        None if inp_cpu.k_scale is None else inp_cpu.k_scale[sl],
                        None if inp_cpu.v_scale is None else inp_cpu.v_scale[sl])


def oracle_us(inp_cpu, threads, budget_s=None):
    """Microseconds per whole call of the fp64 oracle with `threads` threads.
    Without a budget the whole batch runs as one call; with one, whole
    sequences run one by one until the budget is spent and the time is
    scaled by the batch's algorithmic bytes over the sample's.  Returns
    (us, sample text)."""
    import oracle
    oracle.set_threads(threads)
    B = inp_cpu.q.shape[0]
    total = algorithmic_bytes(inp_cpu)
    if budget_s is None:
        t0 = time.perf_counter()
        oracle_call(inp_cpu, slice(0, B))
        return 1e6 * (time.perf_counter() - t0), "whole call"
    t_used, done, seqs = 0.0, 0, 0
    while seqs < B and (seqs == 0 or t_used < budget_s):
        sl = slice(seqs, seqs + 1)
        t0 = time.perf_counter()
        oracle_call(inp_cpu, sl)
        t_used += time.perf_counter() - t0
        sub = sub_inputs(inp_cpu, sl)
        done += algorithmic_bytes(sub)
        seqs += 1
    if seqs == B:
        return 1e6 * t_used, "whole batch, sequence by sequence"
    return 1e6 * t_used * total / done, "%d of %d sequences, scaled by bytes" % (seqs, B)


# The five reference workloads (1000-position dense, MTP verify, the ragged
# batch, top-k gather, int8 at 131072 positions) with their tags in the bench
# line.
BASELINE_CONFIGS = (("c1_dense_1k", "dense_1k"), ("c2_mtp_verify", "mtp_verify"),
                    ("c3_ragged", "ragged"), ("c4_gather", "gather"), ("c5_int8", "int8"))


def baseline_configs(device, stream, peak, kernel, with_cpu=True, cpu_budget=8.0):
    """The five named workloads: GPU us per call (mean, median, min, p90 over
    individually timed replays of a 10-call graph), KV GB/s and fraction of
    the peak, and the fp64 oracle's us per call on the host cores with every
    core and with one.  The int8 workload's oracle runs once per thread
    count (one of its four sequences with one thread, scaled); the ragged
    workload's one-thread run takes whole sequences for about cpu_budget
    seconds."""
    from decode_attention_preallocated_gb300 import workloads as W
    cores = len(os.sched_getaffinity(0))
    res = {}
    for tag, name in BASELINE_CONFIGS:
        inp = W.workload(name, seed=1, device=device)
        ws = workspace_for(inp, device)
        out = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=device)
        fn = call_fn(inp, out, ws, kernel)
        for _ in range(5):
            fn()
        st = time_stats(fn, stream, calls=10, replays=10 if name in ("ragged", "int8") else 20)
        nb = algorithmic_bytes(inp)
        e = {"us": round(st["mean"], 2), "med": round(st["median"], 2),
             "min": round(st["min"], 2), "p90": round(st["p90"], 2),
             "GBps": round(nb / st["mean"] / 1e3, 1),
             "frac": round(nb / st["mean"] / 1e3 / peak, 4)}
        ws.close()
        if with_cpu:
            ci = cpu_view(inp)
            big = name in ("ragged", "int8")
            us_n, _ = oracle_us(ci, cores)
            us_1, how = oracle_us(ci, 1, (cpu_budget if name == "ragged" else 0.0) if big else None)
            e["cpu_us"] = round(us_n, 1)
            e["cpu1_us"] = round(us_1, 1)
            if big:
                e["cpu1_sample"] = how
            del ci
        res[tag] = e
        del inp, out
        torch.cuda.empty_cache()
    for cap in (3000, 131072):
        inp = W.dense_inputs(1, 4, 16, 4, 256, cap, [3000], 1, True, device=device)
        ws = workspace_for(inp, device)
        out = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=device)
        fn = call_fn(inp, out, ws, kernel)
        for _ in range(5):
            fn()
        res["c2_mtp_verify"]["cap%d_us" % cap] = round(time_stats(fn, stream)["mean"], 2)
        ws.close()
        del inp, out
    res["cpu"] = {"cores": cores, "model": cpu_model()}
    return res


# --------------------------------------------------------------- the arms
def run_reference(args):
    rank, world, local = rank_info()
    if world > 1 and rank != 0:
        return 0
    from decode_attention_preallocated_gb300 import workloads as W
    inp = W.workload(WORKLOAD, seed=1, device="cpu")
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    # one step = the oracle on one whole sequence of the batch (bounded sample)
    per_step = []
    steps = max(1, args.steps)
    warm = max(0, min(args.warmup, 1))
    B = inp.q.shape[0]
    total_bytes, total_t = 0, 0.0
    for s in range(warm + steps):
        b = s % B
        sl = slice(b, b + 1)
        t0 = time.perf_counter()
        oracle.dense(inp.q[sl], inp.k[sl], inp.v[sl], [inp.lengths_host[b]], inp.n_q,
                     inp.causal, inp.scale)
        dt = time.perf_counter() - t0
        if s >= warm:
            nb = kv_bytes([inp.lengths_host[b]], inp.k.shape[1], inp.q.shape[3], 2)
            total_bytes += nb
            total_t += dt
            per_step.append(dt)
    value = total_bytes / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_t / steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "step": "fp64 oracle over one whole sequence "
                   "of the batch (all 16 heads x 6 rows)", "l2": "host run"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle",
                         "sample": "%d whole sequence(s), round-robin over the batch" % steps},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def extras(args, device, stream, peak, kernel):
    """Per-mode timings beside the headline: the next rows' workloads, the
    gather's capacity sweep and the depth sweep (µs/call and GB/s from CUDA
    graph replay; us_python_loop: the same calls launched one by one from
    Python, which host overhead bounds for the small workloads)."""
    from decode_attention_preallocated_gb300 import fd
    from decode_attention_preallocated_gb300 import workloads as W
    res = {}

    def measure(tag, inp, n=200):
        ws = workspace_for(inp, device)
        out = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=device)
        fn = call_fn(inp, out, ws, kernel)
        for _ in range(5):
            fn()
        ms_host = time_calls(fn, n, stream)         # each call launched from Python
        calls = min(n, GRAPH_CALLS)
        g = capture(fn, calls, stream)
        ms = time_graph(g, calls, max(1, n // calls), stream)   # graph replay: GPU time
        del g
        nbytes = algorithmic_bytes(inp)
        res[tag] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                    "frac": round(nbytes / ms / 1e6 / peak, 4), "bytes": nbytes,
                    "us_python_loop": round(ms_host * 1e3, 2)}
        ws.close()

    def measure_fn(tag, fn, nbytes, n=200):
        for _ in range(5):
            fn()
        calls = min(n, GRAPH_CALLS)
        g = capture(fn, calls, stream)
        ms = time_graph(g, calls, max(1, n // calls), stream)
        del g
        res[tag] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                    "frac": round(nbytes / ms / 1e6 / peak, 4), "bytes": nbytes}

    # (the five named workloads are timed by baseline_configs)
    # gather with a per-entry bias (N(0, 2), as a mask-derived list carries)
    inp = W.workload("gather", seed=1, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(3)
    inp.bias = torch.randn(inp.idx.shape, generator=g, device=device) * 2.0
    measure("gather_bias", inp)
    del inp
    # the gather workload over an int8 cache (per-cell fp32 scales)
    inp = W.gather_inputs(1, 1, 32, 4, 128, 131072, 2048, 128, 1, device=device, int8=True)
    measure("gather_int8", inp)
    del inp
    # the same selection as a mask over the whole window (hidden 32-position
    # chunks not read), and masks that leave 5 % / 25 % / all of the chunks
    # visible; bytes: the visible chunks' K / V rows.  The tensor-core kernel
    # lists the visible chunks first (the workspace has room); "_in_place"
    # gives it a workspace sized for the call alone, so each tile of the
    # prefix finds its chunks itself.
    inp = W.workload("gather", seed=1, device=device)
    ws_m = workspace_for(inp, device)
    rows_m = inp.q.shape[2] // inp.k.shape[1]
    G_m = fd.auto_num_ctas(fd.FD_KERNEL_TC, inp.q.shape[3], fd.FD_BF16, rows_m, 0)
    ws_t = fd.Workspace(inp.k.shape[1], rows_m, inp.q.shape[3], G_m, device=device)
    out_m = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=device)
    cap = inp.k.shape[2]
    for tag, keep in (("masked_gather_list_131k", None), ("masked_5pct_131k", 0.05),
                      ("masked_25pct_131k", 0.25), ("masked_100pct_131k", 1.0)):
        mask = torch.full((1, 1, cap), -float("inf"), device=device)
        if keep is None:
            mask[0, 0, inp.idx[0, 0].long()] = 0.0
        else:
            gm = torch.Generator(device=device)
            gm.manual_seed(9)
            live = torch.rand(cap // 32, generator=gm, device=device) < keep
            mask.view(1, 1, -1, 32)[0, 0, live] = 0.0
        chunks = int((mask.view(-1, 32) != -float("inf")).any(1).sum())
        nbytes = chunks * 32 * inp.k.shape[1] * inp.q.shape[3] * 4
        measure_fn(tag, lambda: fd.decode_masked(
            inp.q, inp.k, inp.v, inp.kv_lengths, mask, n_q=1, causal=False, scale=inp.scale,
            out=out_m, workspace=ws_m, kernel=kernel), nbytes, 50)
        res[tag]["visible_chunks"] = chunks
        if keep in (None, 0.05):
            measure_fn(tag + "_in_place", lambda: fd.decode_masked(
                inp.q, inp.k, inp.v, inp.kv_lengths, mask, n_q=1, causal=False,
                scale=inp.scale, out=out_m, workspace=ws_t, kernel=kernel, num_ctas=G_m),
                nbytes, 50)
    ws_m.close()
    ws_t.close()
    del inp, mask
    # gather: time follows the list length, not the capacity
    for K in (512, 2048, 8192):
        for cap in (8192, 32768, 131072):
            inp = W.gather_inputs(1, 1, 32, 4, 128, cap, K, 128, 1, device=device)
            measure("gather_K%d_cap%d" % (K, cap), inp, 100)
            del inp
    torch.cuda.empty_cache()
    # fused append: the MTP-verify and ragged workloads as one step that
    # writes the window's rows (4 / 6 per sequence) and attends
    for name in ("mtp_verify", "ragged"):
        inp = append_inputs(name, 1, device)
        measure("append_" + name, inp, 200 if name == "mtp_verify" else 50)
        del inp
        torch.cuda.empty_cache()
    # int8 caches with 64 rows per kv head (4 causal rows x 16 heads), which
    # the tensor-core kernel serves in two parts of 32 rows
    for d in (128, 256):
        tag = "int8_rows64_d%d" % d
        try:
            inp = W.dense_inputs(4, 4, 64, 4, d, 32768, [32768] * 4, 5, True, device=device,
                                 int8=True)
            measure(tag, inp, 50)
        except Exception as e:   # an extra: recorded, never fatal to the line
            res[tag] = {"error": repr(e)[:200]}
        inp = None
        torch.cuda.empty_cache()
    # paged caches: the ragged and int8 workloads with their pages scattered
    # over a pool (bytes: the same K/V rows as the flat caches)
    for name in ("paged_ps16", "paged_ps64", "paged_ps256", "paged_int8_ps64",
                 "paged_int8_ps256"):
        inp = W.workload(name, seed=1, device=device)
        measure(name, inp, 50)
        del inp
        torch.cuda.empty_cache()
    # block top-k selection (gather lists from block scores), alone and
    # followed by the gather it feeds
    for tag, B, n_q, nb, bs, k in (("topk_131k_1row", 1, 1, 2048, 64, 32),
                                   ("topk_32k_48rows", 8, 6, 512, 64, 32),
                                   ("topk_2m_1row", 1, 1, 32768, 64, 32)):
        g = torch.Generator(device=device)
        g.manual_seed(5)
        scores = torch.randn((B, n_q, nb), generator=g, device=device)
        lens = torch.full((B,), nb * bs, dtype=torch.int32, device=device)
        idx = torch.empty((B, n_q, k * bs), dtype=torch.int32, device=device)
        measure_fn(tag, lambda: fd.topk_blocks(scores, lens, bs, k, out=idx),
                   scores.numel() * 4 + idx.numel() * 4)
    inp = W.dense_inputs(1, 1, 32, 4, 128, 131072, [131072], 1, False, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(6)
    scores = torch.randn((1, 1, 2048), generator=g, device=device)
    idx = torch.empty((1, 1, 2048), dtype=torch.int32, device=device)
    out_g = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=device)
    ws_g = workspace_for(inp, device)

    def select_gather():
        fd.topk_blocks(scores, inp.kv_lengths, 64, 32, out=idx)
        fd.decode_gather(inp.q, inp.k, inp.v, idx, scale=inp.scale, out=out_g, workspace=ws_g,
                         kernel=kernel)

    measure_fn("select_gather_131k_32q4kv", select_gather,
               2048 * 4 * 2 + 2048 * 4 * 128 * 2 * 2)
    ws_g.close()
    measure("dense_scan_131k_32q4kv", inp, 50)
    del inp
    for L in (32768, 65536, 131072):
        for (Hq, Hkv, d, n_q, B) in ((16, 4, 256, 6, 8), (16, 4, 256, 1, 4), (8, 2, 128, 1, 8)):
            inp = W.dense_inputs(B, n_q, Hq, Hkv, d, L + 1000, [L] * B, 100, n_q > 1,
                                 device=device)
            measure("sweep_L%d_B%d_%dq%dkv_d%d_nq%d" % (L, B, Hq, Hkv, d, n_q), inp, 30)
            del inp
            torch.cuda.empty_cache()
    return res


def run_fd(args):
    from decode_attention_preallocated_gb300 import build as fdbuild
    from decode_attention_preallocated_gb300 import fd

    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    fdbuild.build()
    fd.lib()
    kernel = {"auto": fd.FD_KERNEL_AUTO, "simt": fd.FD_KERNEL_SIMT,
              "tc": fd.FD_KERNEL_TC}[args.kernel]
    peak, peak_kind = peaks()

    inp = make_inputs(args.workload, seed=1 + rank, device=device)
    nbytes = algorithmic_bytes(inp)
    ws = workspace_for(inp, device)
    out = torch.empty(inp.q.shape, dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device)
    fn = call_fn(inp, out, ws, kernel)

    warm = max(3, args.warmup)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
    torch.cuda.synchronize()
    steps = args.steps
    if steps <= 0:   # auto: about 3 s of timed work so the clock samples mean something
        ms = time_calls(fn, 5, stream)
        steps = int(max(20, min(20000, 3000.0 / max(ms, 1e-3))))
    # the timed steps run as replays of a captured graph of calls
    gcalls = max(1, min(GRAPH_CALLS, steps))
    replays = -(-steps // gcalls)
    steps = replays * gcalls
    graph = capture(fn, gcalls, stream)
    with torch.cuda.stream(stream):
        graph.replay()          # untimed: the graph's first launch uploads it
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local])
    barrier()
    sampler.start()
    time.sleep(0.25)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(replays):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier()
    clocks = sampler.stop()
    ms_step = ev0.elapsed_time(ev1) / steps
    ms_max = max_over_ranks(ms_step, world, device)
    all_bytes = nbytes * world
    value = aggregate_gbs(nbytes, world, ms_max)

    # end to end through the public call with host buffers: every step copies
    # q, both caches, kv_lengths (and the scales, index lists or block table
    # the workload has) from pinned host memory, decodes, and reads the output
    # back
    names = [n for n in ("q", "k", "v", "kv_lengths", "k_scale", "v_scale", "idx", "block_table",
                         "k_new", "v_new") if getattr(inp, n, None) is not None]
    host = {} if args.no_e2e else {n: getattr(inp, n).cpu().pin_memory() for n in names}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        for n, x in host.items():
            getattr(inp, n).copy_(x, non_blocking=True)
        fn()
        out_host.copy_(out, non_blocking=True)

    e2e_value = None
    if not args.no_e2e:
        e2e_steps = max(3, min(20, steps))
        with torch.cuda.stream(stream):
            e2e_step()
        barrier()
        e_ms = time_calls(e2e_step, e2e_steps, stream)
        e2e_value = round(aggregate_gbs(nbytes, world, max_over_ranks(e_ms, world, device)), 3)

    result = None
    if rank == 0:
        achieved = nbytes / (ms_step * 1e-3) / 1e9
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu_inp = cpu_view(inp)
            gbs, cores, sample = oracle_sample(cpu_inp, budget_s=args.cpu_budget)
            cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                   "sample": sample, "cpu_model": cpu_model()}
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(args.workload), "seed": 1,
                       "kv_lengths": inp.lengths_host,
                       "kv_bytes_per_step": nbytes, "us_per_call": round(ms_step * 1e3, 2),
                       "l2": "inputs larger than L2 (no flush)",
                       "launch": "CUDA graph of %d calls, replayed %d times" % (gcalls, replays),
                       "parallelism": "replicas (one batch per GPU, no collective)",
                       "kernel": args.kernel},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": recorded_traffic(args.workload),
                         "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                         if peak_kind == "measured" else "fallback 6.8 TB/s"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clocks,
            "gpu_launches": steps,
        }
        if not args.no_extras and world == 1:
            result["modes"] = extras(args, device, stream, peak, kernel)
        if not args.no_configs and world == 1:
            # last in the line, so that a tail of it keeps every named workload
            result["configs"] = baseline_configs(device, stream, peak, kernel,
                                                 not args.no_cpu_baseline, args.cpu_budget)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    ws.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="0 = auto (~3 s timed)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["fd", "reference"], default="fd")
    ap.add_argument("--kernel", choices=["auto", "simt", "tc"], default="auto")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="ragged (default), dense_1k, mtp_verify, gather, int8, "
                         "or sweep:L,B,Hq,Hkv,d,n_q")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload block (GPU stats and oracle timings)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_fd(args)


if __name__ == "__main__":
    sys.exit(main())
