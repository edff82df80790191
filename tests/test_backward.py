"""attn_fwd_lse and attn_bwd (the tcgen05 dK/dV and dQ passes, through the C
ABI) against the float64 oracle: the log-sum-exps, and dq, dk, dv at sizes
the oracle finishes in seconds (ragged tails, GQA/MQA, windows, non-causal,
more items than SMs), sampled rows and keys at the full workload size, plus
determinism, a NaN canary and the S = 1 closed form.

Tolerance of the gradients: the kernels round P and dS to bf16 before their
MMAs and the outputs to bf16 (a relative error of at most 2^-8 each), and D_i
comes from the bf16-rounded forward output; every sum is fp32.  Unlike the
forward output (a convex combination of value rows, so bounded by them), a
gradient entry can be large, and the rounding of the result alone reaches
2^-8 of it.  The bar is therefore the forward's bar plus one bf16 rounding of
the result: element-wise |err| <= 2e-2 + 2^-8 |ref|, and mean |err| <=
2e-3 + 2^-8 mean |ref|.  Measured on every case below (GB300): the largest
|err| - 2^-8 |ref| is 1.34e-2 (two thirds of the absolute term) and the
largest mean |err| 1.47e-3 (with CHS_ERROR_TABLE set, every comparison
appends its errors to that file).
"""
import json
import os

import numpy as np
import pytest
import torch

import causal_head_self_gb300 as chs
import oracle
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs
from parity import sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()


def _close_scaled(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if not ref.size:
        return
    err = np.abs(got - ref)
    if os.environ.get("CHS_ERROR_TABLE"):
        # the measured errors behind the bar: max and mean |err|, the
        # reference's RMS, and the largest |err| - 2^-8 |ref| (the error left
        # once one bf16 rounding of the result is taken out)
        with open(os.environ["CHS_ERROR_TABLE"], "a") as f:
            f.write(json.dumps({"case": what, "max_err": float(err.max()),
                                "mean_err": float(err.mean()),
                                "rms_ref": float(np.sqrt(np.mean(ref ** 2))),
                                "max_ref": float(np.abs(ref).max()),
                                "max_err_less_rounding": float(np.max(err - 2.0 ** -8 * np.abs(ref)))})
                    + "\n")
    bound = 2e-2 + 2.0 ** -8 * np.abs(ref)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (f"{what}: |err| {err.flat[worst]:.3e} > {bound.flat[worst]:.3e} "
                                  f"at ref {ref.flat[worst]:.4e}")
    mean_bound = 2e-3 + 2.0 ** -8 * float(np.abs(ref).mean())
    assert err.mean() <= mean_bound, f"{what}: mean|err| {err.mean():.3e} > {mean_bound:.3e}"


def gpu_fwd_bwd(q, k, v, dout, causal, window):
    d = torch.device("cuda")
    q, k, v, dout = q.to(d), k.to(d), v.to(d), dout.to(d)
    o, lse = chs.attn_fwd_lse(q, k, v, causal=bool(causal), window=window)
    dq, dk, dv = chs.attn_bwd(q, k, v, o, dout, lse, causal=bool(causal), window=window)
    assert chs.attn_status() == chs.ATTN_OK
    return o, lse, dq, dk, dv


# ---------------------------------------------------------------- log-sum-exp

@pytest.mark.parametrize("B,Hq,Hkv,S,Dh,causal,window", [
    (1, 2, 2, 300, 128, 1, 0), (2, 4, 2, 257, 64, 1, 33), (1, 2, 1, 200, 128, 0, 0),
    (1, 2, 2, 150, 256, 1, 0)])
def test_lse_matches_oracle_and_output_matches_attn_fwd(B, Hq, Hkv, S, Dh, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=S + Dh)
    d = torch.device("cuda")
    o, lse = chs.attn_fwd_lse(q.to(d), k.to(d), v.to(d), causal=bool(causal), window=window)
    o_plain = chs.attn_fwd(q.to(d), k.to(d), v.to(d), causal=bool(causal), window=window)
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.equal(o, o_plain)
    _, ref = oracle.attention(q, k, v, causal=bool(causal), window=window, return_lse=True)
    # fp32 scores of bf16 inputs: the lse is good to a few fp32 ulps of its terms
    np.testing.assert_allclose(lse.cpu().numpy(), ref, atol=2e-3, rtol=0)


# ---------------------------------------------------------------- gradients

# (B, Hq, Hkv, S, Dh, causal, window)
SMALL = [
    (1, 2, 2, 128, 64, 1, 0),
    (1, 2, 2, 1, 128, 1, 0),
    (1, 2, 2, 2, 64, 1, 0),
    (1, 3, 3, 127, 128, 1, 0),
    (1, 2, 2, 129, 128, 1, 0),
    (2, 2, 2, 300, 64, 1, 0),
    (1, 4, 2, 384, 128, 1, 0),
    (1, 4, 1, 257, 128, 1, 0),
    (1, 2, 2, 300, 128, 0, 0),
    (1, 2, 1, 200, 64, 0, 0),
    (1, 4, 2, 700, 128, 1, 1),
    (1, 4, 2, 700, 128, 1, 17),
    (1, 4, 1, 700, 64, 1, 128),
    (1, 2, 2, 1000, 128, 1, 200),
    (1, 2, 2, 1030, 128, 1, 1000),
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


# more work items than SMs in both passes: barrier phases, stages and the
# accumulators carry from one item into the next
PERSISTENT = [
    (2, 16, 4, 1000, 128, 1, 0),
    (1, 160, 160, 256, 64, 1, 0),
    (2, 12, 12, 700, 128, 1, 300),
    (1, 40, 8, 600, 128, 0, 0),
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
    """S = 1: one weight of 1, so dq = dk = 0 and dv = the group's sum of dout.
    (dS = 1 * (dP - D) with dP = dout . v from the MMA and D = dout . o, o = v,
    from the row reduction: the two fp32 sums differ only in their order, so
    dq and dk are zero up to fp32 rounding of O(10) dot products.)"""
    q, k, v = inputs.prefill_inputs(2, 4, 2, 1, 128, seed=61)
    dout = inputs.grad_inputs(q.shape, seed=61)
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, dout, 1, 0)
    assert float(dq.abs().max()) < 1e-4 and float(dk.abs().max()) < 1e-4
    want = dout.float().reshape(2, 2, 2, 1, 128).sum(2)
    _close_scaled(dv.float().cpu().numpy(), want.numpy(), "dv at S = 1")


def test_deterministic_and_every_output_written():
    q, k, v = inputs.prefill_inputs(1, 6, 2, 333, 128, seed=62)
    dout = inputs.grad_inputs(q.shape, seed=62)
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


def test_rejects_unsupported_head_size_and_aliasing():
    d = torch.device("cuda")
    q = torch.zeros((1, 2, 64, 96), dtype=torch.bfloat16, device=d)
    lse = torch.zeros((1, 2, 64), dtype=torch.float32, device=d)
    with pytest.raises(chs.AttnError) as e:
        chs.attn_bwd(q, q, q, q, q, lse)
    assert e.value.code == chs.ATTN_ERR_UNSUPPORTED
    q = torch.zeros((1, 2, 64, 128), dtype=torch.bfloat16, device=d)
    lse = torch.zeros((1, 2, 64), dtype=torch.float32, device=d)
    with pytest.raises(chs.AttnError) as e:
        chs.attn_bwd(q, q, q, q, q, lse, dq=q)
    assert e.value.code == chs.ATTN_ERR_INVALID_ARG


# ---------------------------------------------------------------- full size

@pytest.mark.parametrize("name,heads", [
    ("backward_mha_b1_h32_s4096_d128", (0, 13, 31)),
    ("backward_gqa_b2_h32kv8_s2048_d128", (4, 5, 6, 7)),   # one whole K/V group
])
def test_workload_sampled(name, heads):
    """The whole workload on the GPU; the oracle on a few heads (a whole K/V
    group, so dk/dv sums are complete), sampled query rows for dq and sampled
    keys for dk/dv (every query row enters those)."""
    w = inputs.WORKLOADS[name]
    q, k, v, dout = inputs.workload_inputs(name)
    _, _, dq, dk, dv = gpu_fwd_bwd(q, k, v, dout, w["causal"], w["window"])
    S, G = w["S"], w["Hq"] // w["Hkv"]
    rows = sample_rows(S, 24, seed=w["seed"], must=(0, 127, 128, S - 1))
    keys = sample_rows(S, 24, seed=w["seed"] + 1, must=(0, 127, 128, S - 1))
    heads = list(heads)
    kv_heads = sorted({h // G for h in heads})
    assert all(h // G in kv_heads for h in heads)
    if G > 1:   # a whole group: every query head of each K/V head taken
        heads = [g * G + j for g in kv_heads for j in range(G)]
    qs, dos = q[:, heads], dout[:, heads]
    ks, vs = k[:, kv_heads], v[:, kv_heads]
    rq, rk, rv = oracle.attention_bwd(qs, ks, vs, dos, causal=w["causal"], window=w["window"],
                                      rows=rows, keys=keys)
    r_t, k_t = torch.from_numpy(rows).cuda(), torch.from_numpy(keys).cuda()
    got_q = dq[:, heads][:, :, r_t].float().cpu().numpy()
    got_k = dk[:, kv_heads][:, :, k_t].float().cpu().numpy()
    got_v = dv[:, kv_heads][:, :, k_t].float().cpu().numpy()
    _close_scaled(got_q, rq, name + " dq")
    _close_scaled(got_k, rk, name + " dk")
    _close_scaled(got_v, rv, name + " dv")
