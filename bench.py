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

def time_oracle(prefill_host, decode_host, w_p, w_d, prefill_heads=None, decode_seqs=None,
                prefill_rows=None, min_prefill_s=0.0):
    """Time the float64 oracle on a sample; returns (sample description,
    prefill TFLOP/s, decode GB/s, seconds, threads).  The prefill sample is
    repeated until it has run for at least min_prefill_s seconds."""
    import oracle
    q, k, v = prefill_host
    B, Hq = w_p["B"], w_p["Hq"]
    heads = prefill_heads or B * Hq
    bsel = [i // Hq for i in range(heads)]
    hsel = [i % Hq for i in range(heads)]
    qs = torch.stack([q[b, h] for b, h in zip(bsel, hsel)])[None]
    ks = torch.stack([k[b, h] for b, h in zip(bsel, hsel)])[None]
    vs = torch.stack([v[b, h] for b, h in zip(bsel, hsel)])[None]
    rows = None if prefill_rows is None else np.arange(w_p["S"] - prefill_rows, w_p["S"])
    q64, k64, v64 = (x.double().numpy() for x in (qs, ks, vs))
    reps, tp = 0, 0.0
    while reps == 0 or tp < min_prefill_s:
        t0 = time.perf_counter()
        oracle.attention(q64, k64, v64, causal=w_p["causal"], window=w_p["window"], rows=rows)
        tp += time.perf_counter() - t0
        reps += 1
    if rows is None:
        pflops = 4 * w_p["Dh"] * heads * visible_pairs(w_p["S"], w_p["causal"], w_p["window"])
    else:
        pflops = 4 * w_p["Dh"] * heads * int(sum(r + 1 for r in rows))
    pflops *= reps
    qd, kc, vc, sl = decode_host
    nseq = decode_seqs or w_d["B"]
    Lmax = int(sl[:nseq].max())
    kc64 = kc[:nseq, :, :Lmax].double().numpy()
    vc64 = vc[:nseq, :, :Lmax].double().numpy()
    q64d = qd[:nseq].double().numpy()
    t0 = time.perf_counter()
    oracle.decode(q64d, kc64, vc64, sl[:nseq].numpy(), window=w_d["window"])
    td = time.perf_counter() - t0
    wd = dict(w_d, B=nseq)
    dbytes = decode_bytes(wd, sl[:nseq].numpy())
    sample = (f"prefill {heads} of {B * Hq} (batch, head) pairs"
              + (f", last {prefill_rows} rows" if rows is not None else ", all rows")
              + (f", {reps} repetitions" if reps > 1 else "")
              + f"; decode {nseq} of {w_d['B']} sequences, all heads")
    return sample, pflops / tp / 1e12, dbytes / td / 1e9, tp + td, oracle.num_threads()


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
    """The oracle on the host cores, as the reference arm."""
    if rank != 0:
        return None
    w_p, w_d = inputs.WORKLOADS[PREFILL], inputs.WORKLOADS[DECODE]
    ph = inputs.workload_inputs(PREFILL)
    dh = inputs.workload_inputs(DECODE)
    # each step: the last `rows` query rows of one head (the costliest rows of
    # a causal pass) and one decode sequence; sized so the run stays short
    budget = max(0.01, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    rows = 64
    _, _, _, sec, _ = time_oracle(ph, dh, w_p, w_d, prefill_heads=1, decode_seqs=1,
                                  prefill_rows=rows)
    while sec < 0.5 * budget and rows < w_p["S"]:
        rows = min(w_p["S"], rows * 2)
        _, _, _, sec, _ = time_oracle(ph, dh, w_p, w_d, prefill_heads=1, decode_seqs=1,
                                      prefill_rows=rows)
    for _ in range(args.warmup):
        time_oracle(ph, dh, w_p, w_d, prefill_heads=1, decode_seqs=1, prefill_rows=rows)
    pv, dv, secs = [], [], 0.0
    for _ in range(args.steps):
        sample, p, d, sec, thr = time_oracle(ph, dh, w_p, w_d, prefill_heads=1, decode_seqs=1,
                                             prefill_rows=rows)
        pv.append(p)
        dv.append(d)
        secs += sec
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
    """Median CUDA-event time (s) of fn() on `stream`, L2 flushed before each."""
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
    return statistics.median(ts)


def chunk_flops(w):
    """4*Dh per visible (query, key) pair of the chunk: row r sees start + r + 1 keys."""
    pairs = sum(w["start"] + r + 1 for r in range(w["Sq"]))
    return 4 * w["Dh"] * w["B"] * w["Hq"] * pairs


PREFILL_CONFIGS = ("prefill_mha_b1_h32_s4096_d128", "prefill_mha_b1_h32_s4096_d128_noncausal",
                   "prefill_gqa_b1_h32kv8_s32768_d128_w4096")


def time_prefill_configs(chs, dev, flush, stream, peaks):
    """The larger prefill shapes beside the headline one (median of 20
    launches after 3 warm-ups, L2 flushed before each): causal MHA at S=4096,
    its non-causal variant, and windowed GQA at S=32768 (window 4096).
    TFLOP/s count only the visible (unmasked) pairs."""
    out = {}
    for name in PREFILL_CONFIGS:
        w = inputs.WORKLOADS[name]
        q, k, v = (x.to(dev) for x in inputs.workload_inputs(name))
        o = torch.empty_like(q)
        t = _time_launches(lambda: chs.attn_fwd(q, k, v, o, causal=bool(w["causal"]),
                                                window=w["window"]), flush, stream)
        tf = prefill_flops(w) / t / 1e12
        out[name] = {"value": tf, "unit": "TFLOP/s", "frac_bf16": tf / peaks["bf16_tflops"],
                     "ms_per_launch": t * 1e3}
        del q, k, v, o
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error while timing the prefill shapes")
    return out


def time_next_rows(chs, dev, flush, stream, peaks):
    """The rows beyond the headline step, each on its own workload (median of
    20 launches after 3 warm-ups, L2 flushed before each): chunked prefill,
    rolling-buffer decode, head size 256 prefill, MQA decode on the tensor
    cores at head sizes 128 and 256, and the backward pass (2.5x the
    forward's FLOPs)."""
    out = {}
    bf16, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]

    name = "chunk_gqa_b2_h32kv8_c1024_at3072_d128"
    w = inputs.WORKLOADS[name]
    q, kc, vc = (x.to(dev) for x in inputs.workload_inputs(name))
    t = _time_launches(lambda: chs.attn_fwd_chunk(q, kc, vc, w["start"]), flush, stream)
    tf = chunk_flops(w) / t / 1e12
    out["F1_chunked_prefill"] = {"workload": name, "value": tf, "unit": "TFLOP/s",
                                 "frac_bf16": tf / bf16, "ms_per_launch": t * 1e3}
    del q, kc, vc

    name = "ring_decode_gqa_b16_h32kv8_c4096_d128"
    w = inputs.WORKLOADS[name]
    q, kc, vc, sl = inputs.decode_inputs(w["B"], w["Hq"], w["Hkv"], w["Tmax"], w["Dh"], w["lmin"],
                                         w["lmax"], w["seed"])
    q, kc, vc, sld = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
    t = _time_launches(lambda: chs.attn_decode_ring(q, kc, vc, sld, window=w["window"]),
                       flush, stream)
    keys = np.minimum(sl.numpy().astype(np.int64), w["window"]).sum()
    by = keys * w["Hkv"] * w["Dh"] * 2 * 2 + 2 * q.numel() * 2 + sl.numel() * 4
    out["F2_ring_decode"] = {"workload": name, "value": by / t / 1e9, "unit": "GB/s",
                             "frac_hbm": by / t / 1e9 / hbm, "tokens_per_s": w["B"] / t,
                             "ms_per_launch": t * 1e3}
    del q, kc, vc, sld

    name = "ring_decode_mqa_b16_h32kv1_c4096_d128"
    w = inputs.WORKLOADS[name]
    q, kc, vc, sl = inputs.decode_inputs(w["B"], w["Hq"], w["Hkv"], w["Tmax"], w["Dh"], w["lmin"],
                                         w["lmax"], w["seed"])
    q, kc, vc, sld = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
    t = _time_launches(lambda: chs.attn_decode_ring(q, kc, vc, sld, window=w["window"]),
                       flush, stream)
    keys = np.minimum(sl.numpy().astype(np.int64), w["window"]).sum()
    by = keys * w["Hkv"] * w["Dh"] * 2 * 2 + 2 * q.numel() * 2 + sl.numel() * 4
    out["F2_ring_decode_mqa"] = {"workload": name, "value": by / t / 1e9, "unit": "GB/s",
                                 "frac_hbm": by / t / 1e9 / hbm, "tokens_per_s": w["B"] / t,
                                 "ms_per_launch": t * 1e3}
    del q, kc, vc, sld

    name = "prefill_gqa_b1_h16kv8_s8192_d256"
    w = inputs.WORKLOADS[name]
    q, k, v = (x.to(dev) for x in inputs.workload_inputs(name))
    t = _time_launches(lambda: chs.attn_fwd(q, k, v), flush, stream)
    tf = prefill_flops(w) / t / 1e12
    out["F3_prefill_d256"] = {"workload": name, "value": tf, "unit": "TFLOP/s",
                              "frac_bf16": tf / bf16, "ms_per_launch": t * 1e3}
    del q, k, v

    name = "decode_mqa_b16_h32kv1_t32768_d128"
    w = inputs.WORKLOADS[name]
    q, kc, vc, sl = inputs.workload_inputs(name)
    by = decode_bytes(w, sl.numpy())
    q, kc, vc, sld = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
    t = _time_launches(lambda: chs.attn_decode(q, kc, vc, sld), flush, stream)
    out["F3_mqa_decode"] = {"workload": name, "value": by / t / 1e9, "unit": "GB/s",
                            "frac_hbm": by / t / 1e9 / hbm,
                            "tflops": decode_flops(w, sl.numpy()) / t / 1e12,
                            "tokens_per_s": w["B"] / t, "ms_per_launch": t * 1e3}
    del q, kc, vc, sld

    name = "decode_mqa_b16_h8kv1_t32768_d256"
    w = inputs.WORKLOADS[name]
    q, kc, vc, sl = inputs.workload_inputs(name)
    by = decode_bytes(w, sl.numpy())
    q, kc, vc, sld = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
    t = _time_launches(lambda: chs.attn_decode(q, kc, vc, sld), flush, stream)
    out["F3_mqa_decode_d256"] = {"workload": name, "value": by / t / 1e9, "unit": "GB/s",
                                 "frac_hbm": by / t / 1e9 / hbm, "tokens_per_s": w["B"] / t,
                                 "ms_per_launch": t * 1e3}
    del q, kc, vc, sld

    name = "backward_mha_b1_h32_s4096_d128"
    w = inputs.WORKLOADS[name]
    q, k, v, do = (x.to(dev) for x in inputs.workload_inputs(name))
    o, lse = chs.attn_fwd_lse(q, k, v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    t = _time_launches(lambda: chs.attn_bwd(q, k, v, o, do, lse, dq, dk, dv), flush, stream)
    fl = 2.5 * 4 * w["Dh"] * w["B"] * w["Hq"] * visible_pairs(w["S"], w["causal"], w["window"])
    out["F4_backward"] = {"workload": name, "value": fl / t / 1e12, "unit": "TFLOP/s",
                          "frac_bf16": fl / t / 1e12 / bf16, "ms_per_launch": t * 1e3,
                          "flops": "2.5 x the forward's (10*Dh per visible pair per head); "
                                   "the kernels execute 14*Dh (S and dP in both passes)"}
    del q, k, v, do, o, lse, dq, dk, dv
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error while timing the next rows")
    return out


def run_gpu(args, rank, world, local_rank):
    import causal_head_self_gb300 as chs
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w_p, w_d = inputs.WORKLOADS[PREFILL], inputs.WORKLOADS[DECODE]
    # weak scaling: every rank runs its own batch (seeds differ per rank)
    qh, kh, vh = inputs.prefill_inputs(w_p["B"], w_p["Hq"], w_p["Hkv"], w_p["S"], w_p["Dh"],
                                       rank_seed(w_p["seed"], rank))
    qdh, kch, vch, slh = inputs.decode_inputs(w_d["B"], w_d["Hq"], w_d["Hkv"], w_d["Tmax"],
                                              w_d["Dh"], w_d["lmin"], w_d["lmax"],
                                              rank_seed(w_d["seed"], rank))
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    o = torch.empty_like(q)
    qd, kc, vc, sl = qdh.to(dev), kch.to(dev), vch.to(dev), slh.to(dev)
    od = torch.empty_like(qd)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    pf, pb = prefill_flops(w_p), prefill_bytes(w_p)
    db, dfl = decode_bytes(w_d, slh.numpy()), decode_flops(w_d, slh.numpy())

    def step(ev=None):
        flush.zero_()
        if ev is not None:
            ev[0].record(stream)
        chs.attn_fwd(q, k, v, o, causal=bool(w_p["causal"]), window=w_p["window"])
        if ev is not None:
            ev[1].record(stream)
        chs.attn_decode(qd, kc, vc, sl, od, window=w_d["window"])
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            step(evs[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    status = chs.attn_status()
    if status != chs.ATTN_OK:
        raise RuntimeError(f"device error in the timed region: {status}")
    t_pre = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3   # seconds
    t_dec = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    t_pre, t_dec, t_wall = max_over_ranks([t_pre, t_dec, t_wall], world, dev)

    # ---------------------------------------------------------- end to end (host buffers)
    e2e_steps = max(3, min(20, args.steps))
    qp, kp, vp = (x.pin_memory() for x in (qh, kh, vh))
    op = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    qdp, kcp, vcp, slp = (x.pin_memory() for x in (qdh, kch, vch, slh))
    odp = torch.empty(od.shape, dtype=od.dtype).pin_memory()
    e2e_p, e2e_d = [], []
    for i in range(e2e_steps + 2):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        flush.zero_()
        e[0].record(stream)
        q.copy_(qp, non_blocking=True)
        k.copy_(kp, non_blocking=True)
        v.copy_(vp, non_blocking=True)
        chs.attn_fwd(q, k, v, o, causal=bool(w_p["causal"]), window=w_p["window"])
        op.copy_(o, non_blocking=True)
        e[1].record(stream)
        qd.copy_(qdp, non_blocking=True)
        kc.copy_(kcp, non_blocking=True)
        vc.copy_(vcp, non_blocking=True)
        sl.copy_(slp, non_blocking=True)
        chs.attn_decode(qd, kc, vc, sl, od, window=w_d["window"])
        odp.copy_(od, non_blocking=True)
        e[2].record(stream)
        torch.cuda.synchronize(dev)
        if i >= 2:
            e2e_p.append(e[0].elapsed_time(e[1]) / 1e3)
            e2e_d.append(e[1].elapsed_time(e[2]) / 1e3)
    if chs.attn_status() != chs.ATTN_OK:
        raise RuntimeError("device error in the end-to-end loop")
    tp_e2e, td_e2e = statistics.mean(e2e_p), statistics.mean(e2e_d)
    tp_e2e, td_e2e = max_over_ranks([tp_e2e, td_e2e], world, dev)
    if rank != 0:
        return None
    del qp, kp, vp, op, qdp, kcp, vcp, slp, odp
    shapes = time_prefill_configs(chs, dev, flush, stream, read_peaks()[0])
    extras = time_next_rows(chs, dev, flush, stream, read_peaks()[0])

    # ---------------------------------------------------------- report
    K = args.steps
    peaks, peak_src = read_peaks()
    traffic = read_traffic()
    pre_launch = t_pre / K
    dec_launch = t_dec / K
    pre_tflops = pf / pre_launch / 1e12
    dec_gbs = db / dec_launch / 1e9
    kp_name = "attn_prefill_sm103a<128>"
    kd_name = "attn_decode_sm103a<128,4>"
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
              "algorithmic_bytes_per_launch": db, "launch_ms": dec_launch * 1e3}
    dominant = roof_d if dec_launch >= pre_launch else roof_p

    # CPU baseline: the oracle on this machine's host cores, N=1 only
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sample, p_tf, d_gbs, sec, thr = time_oracle((qh, kh, vh), (qdh, kch, vch, slh), w_p, w_d,
                                                    min_prefill_s=10.0)
        cpu = {"value": p_tf, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": sample,
               "seconds": sec, "decode_value": d_gbs, "decode_unit": "GB/s"}

    return {
        "impl": "gb300", "metric": METRIC, "value": job_rate(pf, pre_launch, world) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": (t_pre + t_dec) / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{PREFILL} + {DECODE}",
            "prefill": {k: w_p[k] for k in ("B", "Hq", "Hkv", "S", "Dh", "causal", "window")},
            "decode": {k: w_d[k] for k in ("B", "Hq", "Hkv", "Tmax", "Dh", "lmin", "lmax", "window")},
            "l2": "flushed by a 256 MiB write before every step (outside the timed kernels)",
            "parallelism": f"dp{world} (independent batches per GPU)",
        },
        "frac_of_peak": {"prefill_bf16_burst": pre_tflops / peaks["bf16_tflops"],
                         "prefill_bf16_sustained": pre_tflops / peaks["bf16_tflops_sustained"],
                         "decode_hbm": dec_gbs / peaks["hbm_gbs"],
                         "decode_hbm_8TBps_spec": dec_gbs / 8000.0, "peaks": peak_src},
        "decode": {"value": job_rate(db, dec_launch, world) / 1e9, "unit": "GB/s",
                   "tokens_per_s": w_d["B"] * world / dec_launch,
                   "tflops": dfl / dec_launch / 1e12 * world, "ms_per_launch": dec_launch * 1e3},
        "roofline": dominant,
        "rooflines": {"prefill": roof_p, "decode": roof_d},
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(pf, tp_e2e, world) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (qh, kh, vh)),
                "d2h_bytes_per_step": o.numel() * o.element_size(),
                "decode": {"value": job_rate(db, td_e2e, world) / 1e9, "unit": "GB/s",
                           "h2d_bytes_per_step": sum(x.numel() * x.element_size()
                                                     for x in (qdh, kch, vch, slh)),
                           "d2h_bytes_per_step": od.numel() * od.element_size()}},
        "prefill_shapes": shapes,
        "next_rows": extras,
        "gpu_launches": 2 * K,   # one prefill and one decode kernel per step
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
