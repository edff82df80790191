#!/usr/bin/env python
"""Benchmark of the attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. attn_fwd    causal MHA prefill, B=2, 32 heads, S=1024, Dh=128 (the
                 headline workload: hidden 4096 = 32 x 128);
  2. attn_decode one KV-cache decode step, B=16, 32 query / 8 K/V heads,
                 Dh=128, cache lengths uniform in [16384, 32768].
`value` is the prefill throughput in TFLOP/s (4*Dh FLOPs per unmasked
(query, key) pair per query head, masked pairs not counted), whole job over
all ranks.  The decode leg is reported beside it in KV-cache GB/s (every
valid K/V byte counted once, plus q and o) and tokens/s.  L2 is flushed (a
256 MiB write) before every step, outside the timed kernels.

--impl reference times the float64 CPU oracle (the reference the CUDA path
is checked against) on a bounded sample of the same workloads.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from causal_head_self_gb300 import inputs  # noqa: E402

METRIC = "causal attn fwd TFLOP/s & % BF16 peak; decode KV-cache GB/s & % HBM peak"
PREFILL = "prefill_mha_b2_h32_s1024_d128"
DECODE = "decode_gqa_b16_h32kv8_t32768_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------ algorithmic work

def visible_pairs(S, causal, window):
    """Unmasked (query, key) pairs of one head."""
    if not causal:
        return S * S
    if window <= 0 or window >= S:
        return S * (S + 1) // 2
    W = window
    return W * (W + 1) // 2 + (S - W) * W


def prefill_flops(w):
    return 4 * w["Dh"] * w["B"] * w["Hq"] * visible_pairs(w["S"], w["causal"], w["window"])


def prefill_bytes(w):
    """Q, K, V read once and O written once (bf16)."""
    return 2 * w["Dh"] * w["S"] * w["B"] * (2 * w["Hq"] + 2 * w["Hkv"])


def decode_keys(w, seqlens):
    L = np.asarray(seqlens, np.int64)
    if w["window"] > 0:
        L = np.minimum(L, w["window"])
    return int(L.sum())


def decode_bytes(w, seqlens):
    """Every visible cached K and V row once (GQA shares it across the group),
    plus q, o and the lengths."""
    kv = decode_keys(w, seqlens) * w["Hkv"] * w["Dh"] * 2 * 2
    return kv + 2 * w["B"] * w["Hq"] * w["Dh"] * 2 + 4 * w["B"]


def decode_flops(w, seqlens):
    return 4 * w["Dh"] * w["Hq"] * decode_keys(w, seqlens)


# ------------------------------------------------------------------ environment

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def read_traffic():
    """DRAM bytes per launch from a committed ncu summary, kept only while
    the kernel source it was taken from is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for kernel, rec in data.items():
        src = os.path.join(ROOT, rec.get("source", ""))
        try:
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        except OSError:
            continue
        if sha == rec.get("source_sha16"):
            out[kernel] = rec
    return out


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.tmp = False

    def __enter__(self):
        # the raw samples go to $CHS_CLOCKS_CSV when it is set (kept for
        # inspection), otherwise to a temporary file removed after the summary
        keep = os.environ.get("CHS_CLOCKS_CSV")
        if keep:
            self.path = keep.replace("{gpu}", str(self.gpu))
            self.tmp = False
        else:
            fd, self.path = tempfile.mkstemp(prefix=f"clocks_gpu{self.gpu}_", suffix=".csv")
            os.close(fd)
            self.tmp = True
        self.fh = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:   # no nvidia-smi, or no file: the summary reports "unsampled"
            self.proc = None
            if self.fh is not None:
                self.fh.close()
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if self.tmp:
            os.remove(self.path)
            self.path = None
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle timing

def sample_rows(S, n):
    """n query rows spread evenly over 0..S-1 (first and last included).  The
    oracle materialises every full score row, so its cost per row does not
    depend on the row; an even spread also keeps the sample's share of the
    visible (unmasked) pairs close to its share of the rows."""
    n = max(1, min(S, n))
    return np.unique(np.linspace(0, S - 1, n).round().astype(np.int64))


def oracle_prefill_rate(w, host, rows=None, heads=None, min_s=0.0):
    """Time the float64 oracle on a prefill workload `w` (host bf16 q, k, v).
    rows: query rows evaluated per (b, h) (None: all); heads: query heads
    evaluated (None: all; the K/V heads they read are kept).  The call is
    repeated until it has run for min_s seconds.  The whole configuration's
    time is extrapolated linearly in the evaluated rows (the oracle's cost per
    row is constant); returns (TFLOP/s over the configuration's visible
    pairs, seconds spent, sample description)."""
    import oracle
    q, k, v = host
    B, Hq, Hkv, S, Dh = w["B"], w["Hq"], w["Hkv"], w["S"], w["Dh"]
    hsel = list(range(Hq)) if heads is None else list(heads)
    group = Hq // Hkv
    if heads is not None:
        # each chosen query head with its own K/V head: an MHA-shaped sample
        q = q[:, hsel]
        k = k[:, [h // group for h in hsel]]
        v = v[:, [h // group for h in hsel]]
    if rows is None:
        q64 = q.double().numpy()
        rsel = None
        nrows = S
    else:
        rsel = np.asarray(rows, np.int64)
        nrows = rsel.size
        # only the sampled rows are filled (and read); the zero pages of the
        # rest are never touched
        q64 = np.zeros(tuple(q.shape), np.float64)
        q64[:, :, rsel] = q[:, :, torch.from_numpy(rsel)].double().numpy()
    k64, v64 = k.double().numpy(), v.double().numpy()
    reps, t = 0, 0.0
    while reps == 0 or t < min_s:
        t0 = time.perf_counter()
        oracle.attention(q64, k64, v64, causal=w["causal"], window=w["window"], rows=rsel)
        t += time.perf_counter() - t0
        reps += 1
    frac = (len(hsel) / Hq) * (nrows / S)          # share of the (b, h, row) triples run
    t_full = t / reps / frac
    sample = (f"{'all' if heads is None else len(hsel)} of {Hq} query heads x "
              f"{'all' if rows is None else nrows} of {S} rows"
              + (f", {reps} repetitions" if reps > 1 else "")
              + ("" if frac == 1.0 else ", extrapolated linearly in rows"))
    return prefill_flops(w) / t_full / 1e12, t, sample


def oracle_decode_rate(w, host, nseq=None):
    """Time the float64 oracle on a decode step (all heads of the first nseq
    sequences); returns (KV-cache GB/s, seconds, sample description)."""
    import oracle
    qd, kc, vc, sl = host
    n = nseq or w["B"]
    Lmax = int(sl[:n].max())
    kc64 = kc[:n, :, :Lmax].double().numpy()
    vc64 = vc[:n, :, :Lmax].double().numpy()
    q64 = qd[:n].double().numpy()
    t0 = time.perf_counter()
    oracle.decode(q64, kc64, vc64, sl[:n].numpy(), window=w["window"])
    t = time.perf_counter() - t0
    by = decode_bytes(dict(w, B=n), sl[:n].numpy())
    return by / t / 1e9, t, f"{n} of {w['B']} sequences, all heads"


# The oracle beside every configuration of the target: which rows it runs.
CPU_PREFILL_SAMPLES = {
    "prefill_mha_b1_h2_s128_d64": dict(rows=None, heads=None, min_s=0.5),
    "prefill_mha_b2_h32_s1024_d128": dict(rows=None, heads=None, min_s=3.0),
    "prefill_mha_b1_h32_s4096_d128": dict(rows=256, heads=None, min_s=0.0),
    "prefill_mha_b1_h32_s4096_d128_noncausal": dict(rows=256, heads=None, min_s=0.0),
    "prefill_gqa_b1_h32kv8_s32768_d128_w4096": dict(rows=64, heads=None, min_s=0.0),
}


def cpu_baseline_all(prefill_host=None, decode_host=None):
    """The float64 oracle on this machine's host cores for every configuration:
    the two small prefills whole (repeated), the S=4096 prefills on 256 rows
    per head and the S=32768 windowed prefill on 64 rows per head (each
    extrapolated linearly in rows), the decode step whole."""
    import oracle
    out = {}
    for name, smp in CPU_PREFILL_SAMPLES.items():
        w = inputs.WORKLOADS[name]
        host = prefill_host if (prefill_host is not None and name == PREFILL) \
            else inputs.workload_inputs(name)
        rows = None if smp["rows"] is None else sample_rows(w["S"], smp["rows"])
        tf, sec, sample = oracle_prefill_rate(w, host, rows=rows, heads=smp["heads"],
                                              min_s=smp["min_s"])
        out[name] = {"value": tf, "unit": "TFLOP/s", "seconds": sec, "sample": sample}
        del host
    wd = inputs.WORKLOADS[DECODE]
    host = decode_host if decode_host is not None else inputs.workload_inputs(DECODE)
    gbs, sec, sample = oracle_decode_rate(wd, host)
    out[DECODE] = {"value": gbs, "unit": "GB/s", "seconds": sec, "sample": sample}
    return out, oracle.num_threads()


# ------------------------------------------------------------------ arms

# ------------------------------------------------------------------ ranks (N > 1)

def rank_seed(seed, rank):
    """Weak scaling: every rank runs its own, independent batch."""
    return seed + 1000 * rank


def max_over_ranks(values, world, device=None):
    """The slowest rank's times (the job ends when it does); identity at N=1."""
    if world <= 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_rate(work_per_rank, seconds_slowest, world):
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return work_per_rank * world / seconds_slowest


def run_reference(args, rank, world):
    """The oracle on the host cores, as the reference arm: each step runs the
    headline prefill on query rows spread evenly over the sequence (all
    heads) and the decode step on one sequence; the row count is sized so the
    whole run stays within a few minutes."""
    if rank != 0:
        return None
    w_p, w_d = inputs.WORKLOADS[PREFILL], inputs.WORKLOADS[DECODE]
    ph = inputs.workload_inputs(PREFILL)
    dh = inputs.workload_inputs(DECODE)
    budget = max(0.02, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    n = 16
    _, sec, _ = oracle_prefill_rate(w_p, ph, rows=sample_rows(w_p["S"], n))
    while sec < 0.5 * budget and n < w_p["S"]:
        n = min(w_p["S"], n * 2)
        _, sec, _ = oracle_prefill_rate(w_p, ph, rows=sample_rows(w_p["S"], n))
    rows = None if n >= w_p["S"] else sample_rows(w_p["S"], n)

    def one_step():
        tf, tp, sample = oracle_prefill_rate(w_p, ph, rows=rows)
        gbs, td, dsample = oracle_decode_rate(w_d, dh, nseq=1)
        return tf, gbs, tp + td, f"prefill {sample}; decode {dsample}"

    for _ in range(args.warmup):
        one_step()
    pv, dv, secs, sample = [], [], 0.0, ""
    for _ in range(args.steps):
        tf, gbs, sec, sample = one_step()
        pv.append(tf)
        dv.append(gbs)
        secs += sec
    import oracle
    thr = oracle.num_threads()
    value = statistics.median(pv)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{PREFILL} + {DECODE}", "sample_per_step": sample},
        "decode": {"value": statistics.median(dv), "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _time_launches(fn, flush, stream, iters=20, warmup=3):
    """Latency of one isolated launch: fn() between two CUDA events on
    `stream`, L2 flushed (a 256 MiB write) before each, synchronised after
    each.  Returns {median, min, max, mean} in seconds over `iters` launches."""
    for _ in range(warmup):
        fn()
    ts = []
    for _ in range(iters):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    return {"median": statistics.median(ts), "min": min(ts), "max": max(ts),
            "mean": statistics.mean(ts)}


def _time_throughput(fns, stream, iters=20, warmup=3, graph=True):
    """Mean time (s) per launch of `iters` launches back to back on `stream`,
    launch i running fns[i % len(fns)] (each on its own copy of the inputs),
    bracketed by one pair of CUDA events.  With `graph`, the same launches
    are captured in one CUDA graph and the graph is replayed between the
    events, so that the host's cost per call (Python binding, argument
    checks, launch calls: about 13-15 us) does not set the rate of launches
    shorter than it; returns (graph time, eager time), else the eager time."""
    for i in range(warmup):
        fns[i % len(fns)]()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(iters):
        fns[i % len(fns)]()
    e1.record(stream)
    torch.cuda.synchronize()
    eager = e0.elapsed_time(e1) / 1e3 / iters
    if not graph:
        return eager
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(iters):
            fns[i % len(fns)]()
    g.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    captured = e0.elapsed_time(e1) / 1e3 / iters
    del g
    return captured, eager


def input_sets(set_bytes, l2_bytes, cap=16):
    """Copies of a launch's inputs to cycle through so that a copy is read
    again only after at least four L2 capacities of other data have passed:
    every launch then reads its inputs from DRAM, without a flush."""
    return max(1, min(cap, math.ceil(4 * l2_bytes / max(1, set_bytes))))


def _nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts)


def _copies(n, *ts):
    """n sets of device tensors: the given ones, then n - 1 clones."""
    return [tuple(ts)] + [tuple(t.clone() for t in ts) for _ in range(n - 1)]


def _packed(ts, dev):
    """((pinned host buffer, device buffer), device views): the tensors ts back
    to back (each at a 256-byte boundary) in one pinned host buffer, and views
    of the same layout into one device buffer of that size."""
    offs, n = [], 0
    for t in ts:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(n, dtype=torch.uint8).pin_memory()
    devbuf = torch.empty(n, dtype=torch.uint8, device=dev)
    views = []
    for t, off in zip(ts, offs):
        nb = t.numel() * t.element_size()
        host[off:off + nb].view(t.dtype).view(t.shape).copy_(t)
        views.append(devbuf[off:off + nb].view(t.dtype).view(t.shape))
    return (host, devbuf), views


def _pipelined_e2e(dev, stream, host_in, dev_in, run, dev_out, host_out, steps):
    """Seconds per step of `steps` end-to-end steps pipelined over two device
    buffer sets: step i's inputs cross to the device (a copy stream) while
    step i-1 computes (on `stream`) and step i-2's result crosses back (a
    second copy stream).  Every step copies its inputs in and its result out
    inside the timed region; the buffers alternate, and each copy or launch
    waits for the last use of the buffer it overwrites."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    t0.record(s_in)
    for i in range(steps):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])      # step i-2's launch has read dev_in[b]
            dev_in[b].copy_(host_in, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])         # step i-2's result has left dev_out[b]
        run(b)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            host_out[b].copy_(dev_out[b], non_blocking=True)
            ev_out[b].record(s_out)
    s_out.wait_event(ev_in[(steps - 1) % 2])
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    return t0.elapsed_time(t1) / 1e3 / steps


def _row(work, unit, per_launch, lat, peak=None, eager=None, **extra):
    """One timed row: throughput from back-to-back launches (replayed from a
    CUDA graph; `eager`: the same launches issued from Python), latency beside it."""
    val = work / per_launch / (1e12 if unit == "TFLOP/s" else 1e9)
    r = {"value": val, "unit": unit, "ms_per_launch": per_launch * 1e3,
         "latency_isolated_ms": {k: v * 1e3 for k, v in lat.items()}}
    if eager is not None:
        r["ms_per_launch_eager"] = eager * 1e3
    if peak is not None:
        r["frac_bf16" if unit == "TFLOP/s" else "frac_hbm"] = val / peak
    r.update(extra)
    return r


def chunk_flops(w):
    """4*Dh per visible (query, key) pair of the chunk: row r sees start + r + 1 keys."""
    pairs = sum(w["start"] + r + 1 for r in range(w["Sq"]))
    return 4 * w["Dh"] * w["B"] * w["Hq"] * pairs


LEAD_SLEEP_CYCLES = 400_000   # about 0.2 ms at the GB300's clocks

PREFILL_CONFIGS = ("prefill_mha_b1_h32_s4096_d128", "prefill_mha_b1_h32_s4096_d128_noncausal",
                   "prefill_gqa_b1_h32kv8_s32768_d128_w4096")


def time_prefill_configs(chs, dev, flush, stream, peaks, l2):
    """The larger prefill shapes beside the headline one: causal MHA at
    S=4096, its non-causal variant, and windowed GQA at S=32768 (window
    4096).  Throughput of 20 back-to-back launches over copies of the inputs
    that together exceed L2 (3 warm-ups), and the isolated latency (L2
    flushed before each launch).  TFLOP/s count only the visible pairs."""
    out = {}
    for name in PREFILL_CONFIGS:
        w = inputs.WORKLOADS[name]
        q, k, v = (x.to(dev) for x in inputs.workload_inputs(name))
        o = torch.empty_like(q)
        sets = _copies(input_sets(_nbytes(q, k, v, o), l2), q, k, v, o)
        fns = [lambda s=s: chs.attn_fwd(*s, causal=bool(w["causal"]), window=w["window"])
               for s in sets]
        t, t_eager = _time_throughput(fns, stream)
        lat = _time_launches(fns[0], flush, stream)
        out[name] = _row(prefill_flops(w), "TFLOP/s", t, lat, peaks["bf16_tflops"], eager=t_eager,
                         input_copies=len(sets))
        del q, k, v, o, sets, fns
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error while timing the prefill shapes")
    return out


def _decode_row(chs, name, dev, flush, stream, peaks, l2, ring):
    w = inputs.WORKLOADS[name]
    q, kc, vc, sl = inputs.workload_inputs(name)
    by = decode_bytes(w, sl.numpy())
    qd, kcd, vcd, sld = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
    od = torch.empty_like(qd)
    sets = _copies(input_sets(_nbytes(qd, kcd, vcd), l2), qd, kcd, vcd, sld, od)
    call = chs.attn_decode_ring if ring else chs.attn_decode
    fns = [lambda s=s: call(*s, window=w["window"]) for s in sets]
    t, t_eager = _time_throughput(fns, stream)
    lat = _time_launches(fns[0], flush, stream)
    return _row(by, "GB/s", t, lat, peaks["hbm_gbs"], eager=t_eager, workload=name,
                input_copies=len(sets),
                tokens_per_s=w["B"] / t, tflops=decode_flops(w, sl.numpy()) / t / 1e12)


def time_next_rows(chs, dev, flush, stream, peaks, l2):
    """The rows beyond the headline step, each on its own workload, timed as
    the prefill shapes are: chunked prefill, rolling-buffer decode, head size
    256 prefill, MQA decode on the tensor cores at head sizes 128 and 256,
    decode at head size 64, and the backward pass at head sizes 128 and 256
    (2.5x the forward's FLOPs)."""
    out = {}
    bf16 = peaks["bf16_tflops"]

    name = "chunk_gqa_b2_h32kv8_c1024_at3072_d128"
    w = inputs.WORKLOADS[name]
    q, kc, vc = (x.to(dev) for x in inputs.workload_inputs(name))
    o = torch.empty_like(q)
    sets = _copies(input_sets(_nbytes(q, kc, vc, o), l2), q, kc, vc, o)
    fns = [lambda s=s: chs.attn_fwd_chunk(s[0], s[1], s[2], w["start"], o=s[3]) for s in sets]
    t, t_eager = _time_throughput(fns, stream)
    lat = _time_launches(fns[0], flush, stream)
    out["F1_chunked_prefill"] = _row(chunk_flops(w), "TFLOP/s", t, lat, bf16, eager=t_eager, workload=name,
                                     input_copies=len(sets))
    del q, kc, vc, o, sets, fns

    for key, name, ring in (("F2_ring_decode", "ring_decode_gqa_b16_h32kv8_c4096_d128", True),
                            ("F2_ring_decode_mqa", "ring_decode_mqa_b16_h32kv1_c4096_d128", True),
                            ("F3_mqa_decode", "decode_mqa_b16_h32kv1_t32768_d128", False),
                            ("F3_mqa_decode_d256", "decode_mqa_b16_h8kv1_t32768_d256", False),
                            ("decode_d64", "decode_gqa_b16_h32kv8_t32768_d64", False)):
        out[key] = _decode_row(chs, name, dev, flush, stream, peaks, l2, ring)

    name = "prefill_gqa_b1_h16kv8_s8192_d256"
    w = inputs.WORKLOADS[name]
    q, k, v = (x.to(dev) for x in inputs.workload_inputs(name))
    o = torch.empty_like(q)
    sets = _copies(input_sets(_nbytes(q, k, v, o), l2), q, k, v, o)
    fns = [lambda s=s: chs.attn_fwd(*s) for s in sets]
    t, t_eager = _time_throughput(fns, stream)
    lat = _time_launches(fns[0], flush, stream)
    out["F3_prefill_d256"] = _row(prefill_flops(w), "TFLOP/s", t, lat, bf16, eager=t_eager, workload=name,
                                  input_copies=len(sets))
    del q, k, v, o, sets, fns

    for key, name in (("F4_backward", "backward_mha_b1_h32_s4096_d128"),
                      ("F4_backward_d256", "backward_gqa_b1_h16kv8_s8192_d256")):
        out[key] = _backward_row(chs, name, dev, flush, stream, bf16, l2)
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error while timing the next rows")
    return out


def _backward_row(chs, name, dev, flush, stream, bf16, l2):
    """The backward pass (attn_bwd after attn_fwd_lse) of a named workload."""
    w = inputs.WORKLOADS[name]
    q, k, v, do = (x.to(dev) for x in inputs.workload_inputs(name))
    o, lse = chs.attn_fwd_lse(q, k, v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sets = _copies(input_sets(_nbytes(q, k, v, o, do, dq, dk, dv, lse), l2),
                   q, k, v, o, do, lse, dq, dk, dv)
    fns = [lambda s=s: chs.attn_bwd(*s) for s in sets]
    t, t_eager = _time_throughput(fns, stream)
    lat = _time_launches(fns[0], flush, stream)
    fl = 2.5 * 4 * w["Dh"] * w["B"] * w["Hq"] * visible_pairs(w["S"], w["causal"], w["window"])
    executed = "16*Dh (S in three passes, dP in two)" if w["Dh"] == 256 else \
        "14*Dh (S and dP in both passes)"
    row = _row(fl, "TFLOP/s", t, lat, bf16, eager=t_eager, workload=name, input_copies=len(sets),
               flops="2.5 x the forward's (10*Dh per visible pair per head); "
                     f"the kernels execute {executed}")
    del q, k, v, do, o, lse, dq, dk, dv, sets, fns
    return row


def _host_us_per_call(fn, n=50):
    """Host time of one library call (argument checks, tensor maps, launch),
    with the GPU held busy by a sleep kernel so no call waits on the queue."""
    torch.cuda.synchronize()
    torch.cuda._sleep(100_000_000)
    t0 = time.perf_counter()
    for _ in range(n):
        fn()
    t = (time.perf_counter() - t0) / n
    torch.cuda.synchronize()
    return t * 1e6


def run_gpu(args, rank, world, local_rank):
    import causal_head_self_gb300 as chs
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))
    w_p, w_d = inputs.WORKLOADS[PREFILL], inputs.WORKLOADS[DECODE]
    # weak scaling: every rank runs its own batch (seeds differ per rank)
    qh, kh, vh = inputs.prefill_inputs(w_p["B"], w_p["Hq"], w_p["Hkv"], w_p["S"], w_p["Dh"],
                                       rank_seed(w_p["seed"], rank))
    qdh, kch, vch, slh = inputs.decode_inputs(w_d["B"], w_d["Hq"], w_d["Hkv"], w_d["Tmax"],
                                              w_d["Dh"], w_d["lmin"], w_d["lmax"],
                                              rank_seed(w_d["seed"], rank))
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    o = torch.empty_like(q)
    # the prefill leg cycles through copies of its inputs (64 MiB each) so
    # that every launch reads them from DRAM; the decode cache (2 GiB) is
    # larger than L2 by itself
    psets = _copies(input_sets(_nbytes(q, k, v, o), l2), q, k, v, o)
    qd, kc, vc, sl = qdh.to(dev), kch.to(dev), vch.to(dev), slh.to(dev)
    od = torch.empty_like(qd)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    pf, pb = prefill_flops(w_p), prefill_bytes(w_p)
    db, dfl = decode_bytes(w_d, slh.numpy()), decode_flops(w_d, slh.numpy())

    def prefill(i):
        chs.attn_fwd(*psets[i % len(psets)], causal=bool(w_p["causal"]), window=w_p["window"])

    def decode(i):
        chs.attn_decode(qd, kc, vc, sl, od, window=w_d["window"])

    with ClockSampler(local_rank) as clocks:
        # warm-up steps right before the timed region (no idle gap between
        # them); more of them if W steps are too short to bring the clocks up
        t0 = time.perf_counter()
        warm = 0
        while warm < args.warmup or time.perf_counter() - t0 < 0.3:
            prefill(warm)
            decode(warm)
            warm += 1
            if warm % 8 == 0:
                torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        if chs.attn_status() != chs.ATTN_OK:
            raise RuntimeError("device error during warm-up")
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        # the K steps: their prefills back to back, then their decodes back
        # to back; CUDA events at the start, between the legs and at the end
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        t_wall = time.perf_counter()
        # a short sleep kernel ahead of the first event: the host queues the
        # first launches behind it, so that the timed region does not start
        # with the GPU idle while the host issues the first call (about
        # 10 us, half a prefill launch)
        torch.cuda._sleep(LEAD_SLEEP_CYCLES)
        ev[0].record(stream)
        for i in range(args.steps):
            prefill(i)
        ev[1].record(stream)
        for i in range(args.steps):
            decode(i)
        ev[2].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        if world > 1:
            torch.distributed.barrier()
        status = chs.attn_status()
        if status != chs.ATTN_OK:
            raise RuntimeError(f"device error in the timed region: {status}")
        t_pre = ev[0].elapsed_time(ev[1]) / 1e3   # seconds
        t_dec = ev[1].elapsed_time(ev[2]) / 1e3
        t_pre, t_dec, t_wall = max_over_ranks([t_pre, t_dec, t_wall], world, dev)
        # one isolated launch at a time (L2 flushed before each, an event
        # pair around each): the latency a lone call sees
        lat_p = _time_launches(lambda: prefill(0), flush, stream)
        lat_d = _time_launches(lambda: decode(0), flush, stream)
    host_us = {"attn_fwd": _host_us_per_call(lambda: prefill(0)),
               "attn_decode": _host_us_per_call(lambda: decode(0))}

    # ---------------------------------------------------------- end to end (host buffers)
    # A step's inputs sit back to back in one pinned host buffer and cross to
    # the device in one copy, into one device buffer that q, k and v (and for
    # the decode the cache and the lengths) are views of: one large transfer
    # runs at the host link's rate, several small ones below it.
    e2e_steps = max(3, min(20, args.steps))
    hp, (qe, ke, ve) = _packed((qh, kh, vh), dev)
    op = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hd, (qde, kce, vce, sle) = _packed((qdh, kch, vch, slh), dev)
    odp = torch.empty(od.shape, dtype=od.dtype).pin_memory()
    e2e_p, e2e_d = [], []
    for i in range(e2e_steps + 2):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        flush.zero_()
        e[0].record(stream)
        hp[1].copy_(hp[0], non_blocking=True)
        chs.attn_fwd(qe, ke, ve, o, causal=bool(w_p["causal"]), window=w_p["window"])
        op.copy_(o, non_blocking=True)
        e[1].record(stream)
        hd[1].copy_(hd[0], non_blocking=True)
        chs.attn_decode(qde, kce, vce, sle, od, window=w_d["window"])
        odp.copy_(od, non_blocking=True)
        e[2].record(stream)
        torch.cuda.synchronize(dev)
        if i >= 2:
            e2e_p.append(e[0].elapsed_time(e[1]) / 1e3)
            e2e_d.append(e[1].elapsed_time(e[2]) / 1e3)
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error in the end-to-end loop")
    tp_ser, td_ser = statistics.mean(e2e_p), statistics.mean(e2e_d)
    # the same steps pipelined (a second device buffer set per leg)
    hp2, (qe2, ke2, ve2) = _packed((qh, kh, vh), dev)
    hd2, (qde2, kce2, vce2, sle2) = _packed((qdh, kch, vch, slh), dev)
    o2, od2 = torch.empty_like(o), torch.empty_like(od)
    op2, odp2 = torch.empty_like(op).pin_memory(), torch.empty_like(odp).pin_memory()
    pviews = [(qe, ke, ve, o), (qe2, ke2, ve2, o2)]
    dviews = [(qde, kce, vce, sle, od), (qde2, kce2, vce2, sle2, od2)]
    pipe_steps = max(6, min(40, 2 * args.steps))

    def run_p(b):
        x = pviews[b]
        chs.attn_fwd(x[0], x[1], x[2], x[3], causal=bool(w_p["causal"]), window=w_p["window"],
                     stream=stream)

    def run_d(b):
        x = dviews[b]
        chs.attn_decode(x[0], x[1], x[2], x[3], x[4], window=w_d["window"], stream=stream)

    tp_e2e = _pipelined_e2e(dev, stream, hp[0], [hp[1], hp2[1]], run_p, [o, o2], [op, op2],
                            pipe_steps)
    td_e2e = _pipelined_e2e(dev, stream, hd[0], [hd[1], hd2[1]], run_d, [od, od2], [odp, odp2],
                            pipe_steps)
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error in the pipelined end-to-end loop")
    del hp2, hd2, qe2, ke2, ve2, qde2, kce2, vce2, sle2, o2, od2, op2, odp2, pviews, dviews
    tp_e2e, td_e2e, tp_ser, td_ser = max_over_ranks([tp_e2e, td_e2e, tp_ser, td_ser], world, dev)
    if rank != 0:
        return None
    h2d_p, h2d_d = hp[0].numel(), hd[0].numel()   # bytes per step, padding included
    del hp, hd, qe, ke, ve, qde, kce, vce, sle, op, odp
    peaks, peak_src = read_peaks()
    shapes = time_prefill_configs(chs, dev, flush, stream, peaks, l2)
    extras = time_next_rows(chs, dev, flush, stream, peaks, l2)

    # ---------------------------------------------------------- report
    K = args.steps
    traffic = read_traffic()
    pre_launch = t_pre / K
    dec_launch = t_dec / K
    pre_tflops = pf / pre_launch / 1e12
    dec_gbs = db / dec_launch / 1e9
    # (head size 128 at 1024 keys per head runs on the 64-key-tile kernel)
    kp_name = "attn_prefill_k64_sm103a<128>"
    kd_name = "attn_decode_tc_sm103a<128>"
    roof_p = {"kernel": kp_name, "bound": "tensor", "achieved": pre_tflops,
              "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
              "frac": pre_tflops / peaks["bf16_tflops"],
              "traffic": traffic.get(kp_name, {}).get("bytes_per_launch"),
              "peak_source": f"{peak_src} bf16 burst (kernel timed alone)",
              "algorithmic_flops_per_launch": pf, "launch_ms": pre_launch * 1e3}
    roof_d = {"kernel": kd_name, "bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
              "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
              "traffic": traffic.get(kd_name, {}).get("bytes_per_launch"),
              "peak_source": f"{peak_src} HBM copy bandwidth",
              "algorithmic_bytes_per_launch": db, "launch_ms": dec_launch * 1e3,
              "note": "the leg's time covers the decode kernel and its combine launch"}
    dominant = roof_d if dec_launch >= pre_launch else roof_p

    # CPU baseline: the oracle on this machine's host cores, N=1 only
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        per, thr = cpu_baseline_all((qh, kh, vh), (qdh, kch, vch, slh))
        head = per[PREFILL]
        cpu = {"value": head["value"], "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"{PREFILL}: {head['sample']}; every configuration in per_config",
               "decode_value": per[DECODE]["value"], "decode_unit": "GB/s",
               "seconds": sum(x["seconds"] for x in per.values()), "per_config": per}

    ms = lambda x: {k: v * 1e3 for k, v in x.items()}   # noqa: E731
    return {
        "impl": "gb300", "metric": METRIC, "value": job_rate(pf, pre_launch, world) / 1e12,
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "warmup_steps_run": warm,
        "ms_per_step": (t_pre + t_dec) / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{PREFILL} + {DECODE}",
            "prefill": {k: w_p[k] for k in ("B", "Hq", "Hkv", "S", "Dh", "causal", "window")},
            "decode": {k: w_d[k] for k in ("B", "Hq", "Hkv", "Tmax", "Dh", "lmin", "lmax", "window")},
            "l2": (f"inputs larger than L2: the prefill leg cycles through {len(psets)} copies "
                   f"of its inputs ({len(psets) * _nbytes(q, k, v, o) >> 20} MiB); the decode "
                   f"cache is {_nbytes(kc, vc) >> 20} MiB; no flush inside the timed region"),
            "timing": ("the K steps' prefills back to back, then their decodes back to back, "
                       "CUDA events at the start, between the legs and at the end"),
            "parallelism": f"dp{world} (independent batches per GPU)",
        },
        "frac_of_peak": {"prefill_bf16_burst": pre_tflops / peaks["bf16_tflops"],
                         "prefill_bf16_sustained": pre_tflops / peaks["bf16_tflops_sustained"],
                         "decode_hbm": dec_gbs / peaks["hbm_gbs"],
                         "decode_hbm_8TBps_spec": dec_gbs / 8000.0, "peaks": peak_src},
        "decode": {"value": job_rate(db, dec_launch, world) / 1e9, "unit": "GB/s",
                   "tokens_per_s": w_d["B"] * world / dec_launch,
                   "tflops": dfl / dec_launch / 1e12 * world, "ms_per_launch": dec_launch * 1e3},
        "latency_isolated_ms": {"note": "one launch at a time, L2 flushed before each, "
                                        "an event pair around each (20 launches)",
                                "prefill": ms(lat_p), "decode": ms(lat_d)},
        "host_us_per_call": host_us,
        "roofline": dominant,
        "rooflines": {"prefill": roof_p, "decode": roof_d},
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(pf, tp_e2e, world) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d_p,
                "d2h_bytes_per_step": o.numel() * o.element_size(),
                "ms_per_step": tp_e2e * 1e3,
                "method": f"{pipe_steps} steps pipelined over two device buffer sets (inputs of "
                          "step i cross while step i-1 computes and step i-2's result returns)",
                "serial": {"value": job_rate(pf, tp_ser, world) / 1e12, "unit": "TFLOP/s",
                           "ms_per_step": tp_ser * 1e3,
                           "method": "one step at a time: copy in, launch, copy out, synchronise"},
                "decode": {"value": job_rate(db, td_e2e, world) / 1e9, "unit": "GB/s",
                           "h2d_bytes_per_step": h2d_d,
                           "d2h_bytes_per_step": od.numel() * od.element_size(),
                           "ms_per_step": td_e2e * 1e3,
                           "serial": {"value": job_rate(db, td_ser, world) / 1e9, "unit": "GB/s",
                                      "ms_per_step": td_ser * 1e3}}},
        "prefill_shapes": shapes,
        "next_rows": extras,
        "gpu_launches": 3 * K,   # per step: the prefill kernel, the decode kernel and its combine
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        line = run_gpu(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
