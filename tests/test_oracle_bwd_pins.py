"""Pins of the oracle's backward pass (and of its log-sum-exp) to facts that
do not come from the oracle's own gradient code: the softmax Jacobian values
the textbook page prints, central finite differences of the pinned forward
pass, float64 autograd through a library softmax, and exact identities of
the gradients.  No GPU is needed."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- softmax Jacobian

def test_jacobian_printed_values():
    with open(os.path.join(GOLDEN, "softmax_jacobian.json")) as f:
        g = json.load(f)
    m = []
    for c in g["cases"]:
        J = oracle.softmax_jacobian(c["z"])
        m.append(float(np.abs(J).max()))
        assert abs(m[-1] - c["max_abs_entry"]) <= c["abs_tol"], (c["z"], m[-1])
    assert abs(m[0] / m[1] / g["ratio"] - 1) <= g["ratio_rel_tol"]


def test_jacobian_matches_finite_differences_of_softmax():
    x = _rand(7, 1)
    J = oracle.softmax_jacobian(x)
    eps = 1e-6
    for j in range(x.size):
        e = np.zeros_like(x)
        e[j] = eps
        col = (oracle.softmax(x + e) - oracle.softmax(x - e)) / (2 * eps)
        np.testing.assert_allclose(J[:, j], col, atol=1e-9)
    np.testing.assert_allclose(J.sum(axis=0), 0, atol=1e-15)   # sum_i p_i = 1 for every x


def test_logsumexp_closed_forms_and_brute():
    assert oracle.logsumexp([0.0, -math.inf, 0.0]) == pytest.approx(math.log(2), abs=1e-15)
    assert oracle.logsumexp([-math.inf, -math.inf]) == -math.inf
    x = _rand(9, 2) * 3
    assert oracle.logsumexp(x) == pytest.approx(math.log(sum(math.exp(t) for t in x)), rel=1e-14)
    # a huge shift does not overflow
    assert oracle.logsumexp(x + 1000) == pytest.approx(oracle.logsumexp(x) + 1000, rel=1e-14)


def test_attention_lse_closed_forms():
    """Identical keys: row i sees i+1 equal scores c_i, so lse_i = c_i + log(i+1)
    (with window W: log(min(i+1, W))); a single key: lse = its score."""
    S, Dh = 11, 4
    q = _rand((1, 1, S, Dh), 3)
    k = np.repeat(_rand((1, 1, 1, Dh), 4), S, axis=2)
    v = _rand((1, 1, S, Dh), 5)
    for window in (0, 4):
        _, lse = oracle.attention(q, k, v, causal=True, window=window, return_lse=True)
        c = (q[0, 0] @ k[0, 0, 0]) / math.sqrt(Dh)
        n = np.arange(1, S + 1) if window == 0 else np.minimum(np.arange(1, S + 1), window)
        np.testing.assert_allclose(lse[0, 0], c + np.log(n), rtol=1e-13, atol=1e-13)


def test_attention_lse_against_brute_scores():
    q, k, v = _rand((1, 2, 6, 3), 6), _rand((1, 1, 6, 3), 7), _rand((1, 1, 6, 3), 8)
    _, lse = oracle.attention(q, k, v, causal=True, window=4, return_lse=True)
    for h in range(2):
        for i in range(6):
            s = [float(q[0, h, i] @ k[0, 0, j]) / math.sqrt(3) for j in range(6) if 0 <= i - j < 4]
            assert lse[0, h, i] == pytest.approx(math.log(sum(math.exp(t) for t in s)), rel=1e-13)


# ---------------------------------------------------------------- backward pass

def _loss(q, k, v, dout, **kw):
    """L = sum(dout * o): its gradients are the backward pass given dout."""
    return float((oracle.attention(q, k, v, **kw) * dout).sum())


BWD_CASES = [
    dict(causal=True, window=0, Hq=2, Hkv=2),
    dict(causal=True, window=3, Hq=4, Hkv=2),
    dict(causal=False, window=0, Hq=3, Hkv=1),
    dict(causal=True, window=2, window_p4=True, Hq=2, Hkv=1),
]


@pytest.mark.parametrize("case", BWD_CASES)
def test_backward_matches_central_differences_elementwise(case):
    """Every entry of dq, dk, dv against a central difference of the pinned
    forward pass (tiny sizes: 2 * (numel) forward calls)."""
    case = dict(case)
    Hq, Hkv = case.pop("Hq"), case.pop("Hkv")
    S, Dh = 6, 3
    q, k, v = _rand((1, Hq, S, Dh), 10), _rand((1, Hkv, S, Dh), 11), _rand((1, Hkv, S, Dh), 12)
    dout = _rand((1, Hq, S, Dh), 13)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, **case)
    eps = 1e-5
    for x, grad in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, dout, **case)
            x[idx] = old - eps
            lm = _loss(q, k, v, dout, **case)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, atol=1e-8, rtol=1e-7)


def test_backward_matches_brute_force_directional_difference():
    """A directional derivative of the pure-Python brute-force forward (which
    shares nothing with the C oracle) along a random direction."""
    Hq, Hkv, S, Dh = 2, 1, 5, 2
    q, k, v = _rand((Hq, S, Dh), 20), _rand((Hkv, S, Dh), 21), _rand((Hkv, S, Dh), 22)
    dout = _rand((Hq, S, Dh), 23)
    uq, uk, uv = _rand(q.shape, 24), _rand(k.shape, 25), _rand(k.shape, 26)
    dq, dk, dv = oracle.attention_bwd(q[None], k[None], v[None], dout[None], causal=True, window=3)

    def L(t):
        o = brute.attention((q + t * uq).tolist(), (k + t * uk).tolist(), (v + t * uv).tolist(),
                            causal=True, window=3)
        return float((np.asarray(o) * dout).sum())

    eps = 1e-5
    num = (L(eps) - L(-eps)) / (2 * eps)
    ana = float((dq[0] * uq).sum() + (dk[0] * uk).sum() + (dv[0] * uv).sum())
    assert ana == pytest.approx(num, rel=1e-7, abs=1e-9)


def test_backward_matches_float64_autograd():
    """torch autograd through a library softmax, float64."""
    B, Hq, Hkv, S, Dh, W = 2, 4, 2, 40, 8, 9
    gen = torch.Generator().manual_seed(30)
    q, k, v = (torch.randn(s, generator=gen, dtype=torch.float64)
               for s in ((B, Hq, S, Dh), (B, Hkv, S, Dh), (B, Hkv, S, Dh)))
    dout = torch.randn((B, Hq, S, Dh), generator=gen, dtype=torch.float64)
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    kr, vr = kt.repeat_interleave(Hq // Hkv, 1), vt.repeat_interleave(Hq // Hkv, 1)
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    visible = (j <= i) & (i - j < W)
    s = (qt @ kr.transpose(-1, -2)) / math.sqrt(Dh)
    s = s.masked_fill(~visible, float("-inf"))
    o = torch.softmax(s, -1) @ vr
    o.backward(dout)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal=True, window=W)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12, rtol=1e-10)


def test_backward_identities():
    """sum_j dk_j = 0 (the softmax ignores a shift common to a row's scores:
    adding c to every key adds scale q_i.c to all of row i's scores);
    sum_j dv_j = sum over the group's query heads and rows of dout (weights
    sum to 1); causal row 0 sees one key, so dq_0 = 0; S = 1: dq = dk = 0, dv = dout."""
    B, Hq, Hkv, S, Dh = 2, 6, 2, 33, 5
    q, k, v = _rand((B, Hq, S, Dh), 40), _rand((B, Hkv, S, Dh), 41), _rand((B, Hkv, S, Dh), 42)
    dout = _rand((B, Hq, S, Dh), 43)
    for causal, window in ((True, 0), (True, 7), (False, 0)):
        dq, dk, dv = oracle.attention_bwd(q, k, v, dout, causal=causal, window=window)
        np.testing.assert_allclose(dk.sum(axis=2), 0, atol=1e-12)
        want = dout.reshape(B, Hkv, Hq // Hkv, S, Dh).sum(axis=(2, 3))
        np.testing.assert_allclose(dv.sum(axis=2), want, atol=1e-12)
        if causal:
            np.testing.assert_allclose(dq[:, :, 0], 0, atol=1e-15)
    dq, dk, dv = oracle.attention_bwd(q[:, :, :1], k[:, :, :1], v[:, :, :1], dout[:, :, :1])
    np.testing.assert_allclose(dq, 0, atol=1e-15)
    np.testing.assert_allclose(dk, 0, atol=1e-15)
    np.testing.assert_allclose(dv[:, :, 0], dout[:, :, :1].reshape(B, Hkv, Hq // Hkv, Dh).sum(2),
                               atol=1e-15)


def test_backward_sampled_rows_and_keys_match_full():
    B, Hq, Hkv, S, Dh = 1, 4, 2, 50, 6
    q, k, v = _rand((B, Hq, S, Dh), 50), _rand((B, Hkv, S, Dh), 51), _rand((B, Hkv, S, Dh), 52)
    dout = _rand((B, Hq, S, Dh), 53)
    full = oracle.attention_bwd(q, k, v, dout, window=10)
    rows, keys = [0, 7, 49], [3, 48]
    dq, dk, dv = oracle.attention_bwd(q, k, v, dout, window=10, rows=rows, keys=keys)
    np.testing.assert_array_equal(dq, full[0][:, :, rows])
    np.testing.assert_allclose(dk, full[1][:, :, keys], atol=1e-14)
    np.testing.assert_allclose(dv, full[2][:, :, keys], atol=1e-14)
    dq2, dk2, _ = oracle.attention_bwd(q, k, v, dout, window=10, rows=rows, keys=[])
    np.testing.assert_array_equal(dq2, dq)
    assert dk2.shape == (B, Hkv, 0, Dh)
