"""Run one named workload through the C ABI a few times (for profilers).

    python -m causal_head_self_gb300.run_workload <workload> [--iters N]

Workload names are the keys of causal_head_self_gb300.inputs.WORKLOADS.
Inputs are generated on the host, copied to cuda:0 once, and the kernel
launches run back to back on the current stream; the device status is
checked at the end.
"""
from __future__ import annotations

import argparse
import sys

import torch

import causal_head_self_gb300 as chs
from causal_head_self_gb300 import inputs


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    w = inputs.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    if w["kind"] == "prefill":
        q, k, v = (x.to(dev) for x in inputs.workload_inputs(args.workload))
        o = torch.empty_like(q)
        for _ in range(args.iters):
            chs.attn_fwd(q, k, v, o, causal=bool(w["causal"]), window=w["window"])
    elif w["kind"] == "backward":
        q, k, v, do = (x.to(dev) for x in inputs.workload_inputs(args.workload))
        o, lse = chs.attn_fwd_lse(q, k, v, causal=bool(w["causal"]), window=w["window"])
        for _ in range(args.iters):
            chs.attn_bwd(q, k, v, o, do, lse, causal=bool(w["causal"]), window=w["window"])
    elif w["kind"] == "chunk":
        q, kc, vc = (x.to(dev) for x in inputs.workload_inputs(args.workload))
        for _ in range(args.iters):
            chs.attn_fwd_chunk(q, kc, vc, w["start"], causal=bool(w["causal"]), window=w["window"])
    elif w["kind"] == "ring":
        q, kc, vc, sl = (x.to(dev) for x in inputs.decode_inputs(
            w["B"], w["Hq"], w["Hkv"], w["Tmax"], w["Dh"], w["lmin"], w["lmax"], w["seed"]))
        for _ in range(args.iters):
            chs.attn_decode_ring(q, kc, vc, sl, window=w["window"])
    else:
        q, kc, vc, sl = (x.to(dev) for x in inputs.workload_inputs(args.workload))
        o = torch.empty_like(q)
        for _ in range(args.iters):
            chs.attn_decode(q, kc, vc, sl, o, window=w["window"])
    torch.cuda.synchronize(dev)
    rc = chs.attn_status()
    print(f"{args.workload}: {args.iters} launches, status {chs.error_string(rc)}")
    return 0 if rc == chs.ATTN_OK else 1


if __name__ == "__main__":
    sys.exit(main())
