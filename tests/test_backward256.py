"""attn_bwd at head size 256 (the dV, dK and dQ passes of
backward256_sm103a.cuh, through the C ABI) against the float64 oracle, with
the bar of test_backward.py (the forward's bar plus one bf16 rounding of the
result): ragged tails on the 64- and 128-row block grids, one- and two-token
sequences, GQA/MQA, windows of 1 to 1000 keys, non-causal, more work items
than SMs in every pass, sampled rows and keys at the full Gemma-sized
workload, determinism and a NaN canary."""
import numpy as np
import pytest
import torch

import causal_head_self_gb300 as chs
import oracle
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs
from parity import sample_rows
from test_backward import _close_scaled, gpu_fwd_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()


# (B, Hq, Hkv, S, Dh, causal, window)
SMALL = [
    (1, 2, 2, 64, 256, 1, 0),
    (1, 2, 2, 1, 256, 1, 0),
    (1, 2, 2, 2, 256, 1, 0),
    (1, 2, 2, 63, 256, 1, 0),
    (1, 3, 3, 127, 256, 1, 0),
    (1, 2, 2, 129, 256, 1, 0),
    (2, 2, 2, 300, 256, 1, 0),
    (1, 4, 2, 384, 256, 1, 0),
    (1, 4, 1, 257, 256, 1, 0),
    (1, 2, 2, 300, 256, 0, 0),
    (1, 2, 1, 200, 256, 0, 0),
    (1, 4, 2, 700, 256, 1, 1),
    (1, 4, 2, 700, 256, 1, 17),
    (1, 4, 1, 650, 256, 1, 64),
    (1, 2, 2, 1000, 256, 1, 200),
    (1, 2, 2, 1030, 256, 1, 1000),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,Dh,causal,window", SMALL)
def test_gradients_all_rows_small(B, Hq, Hkv, S, Dh, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=2 * S + Dh + window)
    dout = inputs.grad_inputs(q.shape, seed=S + window)
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, dout, causal, window)
    rq, rk, rv = oracle.attention_bwd(q, k, v, dout, causal=bool(causal), window=window)
    tag = f"{(B, Hq, Hkv, S, Dh, causal, window)}"
    _close_scaled(dv.float().cpu().numpy(), rv, "dv " + tag)
    _close_scaled(dk.float().cpu().numpy(), rk, "dk " + tag)
    _close_scaled(dq.float().cpu().numpy(), rq, "dq " + tag)


# more work items than SMs in every pass: barrier phases, stages and the
# accumulators carry from one item into the next
PERSISTENT = [
    (2, 16, 8, 700, 256, 1, 0),
    (1, 80, 80, 300, 256, 1, 0),
    (1, 48, 12, 500, 256, 1, 150),
    (1, 40, 8, 400, 256, 0, 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,Dh,causal,window", PERSISTENT)
def test_gradients_many_items_per_cta(B, Hq, Hkv, S, Dh, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=3 * S + window)
    dout = inputs.grad_inputs(q.shape, seed=3 * S)
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, dout, causal, window)
    rq, rk, rv = oracle.attention_bwd(q, k, v, dout, causal=bool(causal), window=window)
    tag = f"{(B, Hq, Hkv, S, Dh, causal, window)}"
    _close_scaled(dv.float().cpu().numpy(), rv, "dv " + tag)
    _close_scaled(dk.float().cpu().numpy(), rk, "dk " + tag)
    _close_scaled(dq.float().cpu().numpy(), rq, "dq " + tag)


def test_single_token_closed_form():
    """S = 1: one weight of 1, so dq = dk = 0 and dv = the group's sum of dout."""
    q, k, v = inputs.prefill_inputs(2, 4, 2, 1, 256, seed=71)
    dout = inputs.grad_inputs(q.shape, seed=71)
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, dout, 1, 0)
    assert float(dq.abs().max()) < 1e-4 and float(dk.abs().max()) < 1e-4
    want = dout.float().reshape(2, 2, 2, 1, 256).sum(2)
    _close_scaled(dv.float().cpu().numpy(), want.numpy(), "dv at S = 1")


def test_deterministic_and_every_output_written():
    q, k, v = inputs.prefill_inputs(1, 6, 2, 333, 256, seed=72)
    dout = inputs.grad_inputs(q.shape, seed=72)
    d = torch.device("cuda")
    q, k, v, dout = q.to(d), k.to(d), v.to(d), dout.to(d)
    o, lse = chs.attn_fwd_lse(q, k, v, window=100)
    outs = []
    for _ in range(2):
        dq = torch.full_like(q, float("nan"))
        dk = torch.full_like(k, float("nan"))
        dv = torch.full_like(v, float("nan"))
        chs.attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, window=100)
        assert chs.attn_status() == chs.ATTN_OK
        for t in (dq, dk, dv):
            assert bool(torch.isfinite(t).all())
        outs.append((dq, dk, dv))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_workload_sampled():
    """The Gemma-sized backward (causal GQA, 16 query heads on 8 K/V heads,
    S = 8192) on the GPU; the oracle on one whole K/V group (two query heads)
    at sampled query rows (dq) and sampled keys (dk, dv)."""
    name = "backward_gqa_b1_h16kv8_s8192_d256"
    w = inputs.WORKLOADS[name]
    q, k, v, dout = inputs.workload_inputs(name)
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, dout, w["causal"], w["window"])
    S, G = w["S"], w["Hq"] // w["Hkv"]
    rows = sample_rows(S, 16, seed=w["seed"], must=(0, 63, 64, 127, 128, S - 1))
    keys = sample_rows(S, 16, seed=w["seed"] + 1, must=(0, 63, 64, 127, 128, S - 1))
    kv_heads = [5]
    heads = [g * G + j for g in kv_heads for j in range(G)]
    rq, rk, rv = oracle.attention_bwd(q[:, heads], k[:, kv_heads], v[:, kv_heads], dout[:, heads],
                                      causal=w["causal"], window=w["window"], rows=rows, keys=keys)
    r_t, k_t = torch.from_numpy(rows).cuda(), torch.from_numpy(keys).cuda()
    _close_scaled(dq[:, heads][:, :, r_t].float().cpu().numpy(), rq, name + " dq")
    _close_scaled(dk[:, kv_heads][:, :, k_t].float().cpu().numpy(), rk, name + " dk")
    _close_scaled(dv[:, kv_heads][:, :, k_t].float().cpu().numpy(), rv, name + " dv")
