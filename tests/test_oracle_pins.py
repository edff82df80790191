"""Pins of the float64 oracle to facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print, a closed form, an invariant the pages state, a library routine it
reduces to, or the independent pure-Python brute force.  No GPU is needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from causal_head_self_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _one_head(x):
    return np.asarray(x, np.float64)[None, None]


# ---------------------------------------------------------------- printed values

def test_worked_example_probabilities_and_output():
    """Textbook page, section "Численный пример" (T=3, d_h=2)."""
    g = _golden("worked_example_t3_dh2.json")
    o, p = oracle.attention(_one_head(g["Q"]), _one_head(g["K"]), _one_head(g["V"]),
                            causal=True, return_probs=True)
    half_ulp = 0.5 * 10 ** -g["printed_decimals"]
    np.testing.assert_allclose(p[0, 0], g["P"], atol=half_ulp + 1e-12)
    # the PyTorch printout rounds the exact result to 4 decimals
    np.testing.assert_allclose(o[0, 0], g["O_pytorch"], atol=half_ulp + 1e-12)
    # the hand computation carries rounded weights: agree to the last printed digit
    np.testing.assert_allclose(o[0, 0], g["O_by_hand"], atol=1.5e-4)


def test_worked_example_scores_from_probability_ratios():
    """Unmasked softmax rows recover the printed score table: log(p_j / p_0) = s_j - s_0."""
    g = _golden("worked_example_t3_dh2.json")
    _, p = oracle.attention(_one_head(g["Q"]), _one_head(g["K"]), _one_head(g["V"]),
                            causal=False, return_probs=True)
    s = np.asarray(g["scores_unmasked"])
    got = np.log(p[0, 0] / p[0, 0][:, :1])
    np.testing.assert_allclose(got, s - s[:, :1], atol=1e-4)


def test_exercise_one():
    """Textbook page, section "Вопросы и упражнения", exercise 1."""
    g = _golden("exercise1_t3_dh2.json")
    o, p = oracle.attention(_one_head(g["Q"]), _one_head(g["K"]), _one_head(g["V"]),
                            causal=True, return_probs=True)
    np.testing.assert_allclose(p[0, 0, 2], g["P_row2"], atol=0.5e-4 + 1e-12)
    np.testing.assert_allclose(o[0, 0, 2], g["o_row2"], atol=1e-4)


def test_softmax_printed_rows():
    g = _golden("softmax_rows.json")
    for row in g["rows"]:
        p = oracle.softmax(row["z"])
        if "abs_tol" in row:
            np.testing.assert_allclose(p, row["p"], atol=row["abs_tol"])
        else:
            np.testing.assert_allclose(p, row["p"], rtol=row["rel_tol"])


def test_softmax_masked_entry_is_exactly_zero():
    g = _golden("softmax_rows.json")["masked"]
    z = [float(x) for x in g["z"]]
    p = oracle.softmax(z)
    assert p[g["p_masked_index"]] == 0.0
    assert abs(p.sum() - 1.0) < 1e-15


def test_softmax_mean_max_weight_64_keys():
    """Mean largest weight of 64 random scores: 0.11 at std 1, 0.85 at std 11.3."""
    g = _golden("softmax_rows.json")["mean_max_weight_64_keys"]
    gen = torch.Generator().manual_seed(11)
    z = torch.randn((4000, 64), generator=gen, dtype=torch.float64).numpy()
    for case in g:
        mx = np.mean([oracle.softmax(r * case["score_std"]).max() for r in z])
        assert abs(mx - case["value"]) < case["abs_tol"], (case, mx)


def test_generator_scaled_score_variance():
    """The synthetic inputs have the unit-variance components the scale assumes."""
    g = _golden("scaled_score_variance.json")
    for i, case in enumerate(g["cases"]):
        dh = case["d_h"]
        q, k, _ = inputs.prefill_inputs(1, 1, 1, g["pairs"], dh, seed=100 + i)
        dots = (q[0, 0].double() * k[0, 0].double()).sum(-1).numpy()
        assert abs(dots.var() / case["var_unscaled"] - 1) < g["rel_tol"]
        assert abs((dots / math.sqrt(dh)).var() / case["var_scaled"] - 1) < g["rel_tol"]


# ---------------------------------------------------------------- invariants

def _rand(shape, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=gen, dtype=torch.float64).numpy()


def test_probability_rows_sum_to_one_and_masked_weights_are_zero():
    B, H, S, D = 2, 3, 37, 8
    q, k, v = _rand((B, H, S, D), 1), _rand((B, H, S, D), 2), _rand((B, H, S, D), 3)
    for window in (0, 5):
        _, p = oracle.attention(q, k, v, causal=True, window=window, return_probs=True)
        assert np.all(np.abs(p.sum(-1) - 1.0) < 1e-12)
        i = np.arange(S)[:, None]
        j = np.arange(S)[None, :]
        masked = (j > i) | ((i - j >= window) if window else False)
        assert np.all(p[..., masked] == 0.0)
        assert np.all(p[..., ~masked] > 0.0)


def test_changing_the_last_token_leaves_earlier_rows_unchanged():
    """Causality check of "Multi-head attention in detail" (aigrafen.se): perturb
    the last token, every earlier output row stays bit for bit the same."""
    B, H, S, D = 1, 2, 29, 16
    q, k, v = _rand((B, H, S, D), 4), _rand((B, H, S, D), 5), _rand((B, H, S, D), 6)
    o = oracle.attention(q, k, v, causal=True)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:, :, -1] += 1.0
    k2[:, :, -1] += 1.0
    v2[:, :, -1] += 1.0
    o2 = oracle.attention(q2, k2, v2, causal=True)
    assert np.array_equal(o[:, :, :-1], o2[:, :, :-1])
    assert not np.array_equal(o[:, :, -1], o2[:, :, -1])


def test_single_token_returns_v():
    v = _rand((2, 4, 1, 8), 7)
    o = oracle.attention(_rand((2, 4, 1, 8), 8), _rand((2, 4, 1, 8), 9), v, causal=True)
    np.testing.assert_array_equal(o, v)


def test_identical_keys_give_prefix_mean_of_v():
    """With every key equal, all scores of a row tie and the weights are uniform
    over the visible keys: o_i is the mean of v_j over those keys."""
    S, D = 40, 8
    q = _rand((1, 1, S, D), 10)
    k = np.repeat(_rand((1, 1, 1, D), 11), S, axis=2)
    v = _rand((1, 1, S, D), 12)
    o = oracle.attention(q, k, v, causal=True)
    prefix_mean = np.cumsum(v[0, 0], axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(o[0, 0], prefix_mean, rtol=0, atol=1e-13)
    W = 7
    ow = oracle.attention(q, k, v, causal=True, window=W)
    want = np.stack([v[0, 0, max(0, i - W + 1): i + 1].mean(0) for i in range(S)])
    np.testing.assert_allclose(ow[0, 0], want, rtol=0, atol=1e-13)


def test_constant_v_gives_that_constant():
    S, D = 33, 8
    c = _rand((1, 1, 1, D), 13)
    o = oracle.attention(_rand((1, 2, S, D), 14), _rand((1, 1, S, D), 15),
                         np.repeat(c, S, axis=2), causal=True, window=9)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), atol=1e-13)


def test_gqa_equals_mha_on_heads_repeated_in_group_order():
    """A K/V head shared by a group of H/G query heads equals MHA on K/V heads
    repeated H/G times in a row (repeat_interleave order, g(h) = h // (H/G))."""
    B, Hq, Hkv, S, D = 2, 8, 2, 21, 8
    q = torch.from_numpy(_rand((B, Hq, S, D), 16))
    k = torch.from_numpy(_rand((B, Hkv, S, D), 17))
    v = torch.from_numpy(_rand((B, Hkv, S, D), 18))
    o_gqa = oracle.attention(q, k, v, causal=True)
    rep = Hq // Hkv
    o_mha = oracle.attention(q, k.repeat_interleave(rep, dim=1), v.repeat_interleave(rep, dim=1),
                             causal=True)
    np.testing.assert_array_equal(o_gqa, o_mha)
    # MQA: one K/V head for all query heads
    o_mqa = oracle.attention(q, k[:, :1], v[:, :1], causal=True)
    o_exp = oracle.attention(q, k[:, :1].expand(B, Hq, S, D), v[:, :1].expand(B, Hq, S, D),
                             causal=True)
    np.testing.assert_array_equal(o_mqa, o_exp)


def test_group_size_must_divide():
    q = _rand((1, 6, 4, 4), 19)
    k = _rand((1, 4, 4, 4), 20)
    with pytest.raises(ValueError):
        oracle.attention(q, k, k)


def test_window_conventions_differ_by_one():
    """Section "Скользящее окно": the page's rule 0 <= i-j <= W shows W+1 keys;
    the i-j < W form shows W.  So page(W) == i-j<(W+1)."""
    B, H, S, D = 1, 2, 50, 8
    q, k, v = _rand((B, H, S, D), 21), _rand((B, H, S, D), 22), _rand((B, H, S, D), 23)
    for W in (1, 4, 13):
        a = oracle.attention(q, k, v, causal=True, window=W, window_p4=True)
        b = oracle.attention(q, k, v, causal=True, window=W + 1)
        np.testing.assert_array_equal(a, b)
    # window 1 leaves each query only its own key: o_i = v_i
    np.testing.assert_allclose(oracle.attention(q, k, v, causal=True, window=1), v, atol=1e-15)


def test_decode_equals_last_row_of_full_pass():
    """Section "Prefill и decode": the cached decode step reproduces the last
    row of a full causal pass."""
    B, Hq, Hkv, T, D = 3, 4, 2, 24, 8
    seqlens = np.array([24, 7, 1])
    q = _rand((B, Hq, T, D), 24)
    k, v = _rand((B, Hkv, T, D), 25), _rand((B, Hkv, T, D), 26)
    qd = np.stack([q[b, :, seqlens[b] - 1: seqlens[b]] for b in range(B)])
    od = oracle.decode(qd, k, v, seqlens)
    for b in range(B):
        L = seqlens[b]
        full = oracle.attention(q[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L], causal=True)
        np.testing.assert_allclose(od[b, :, 0], full[0, :, L - 1], rtol=0, atol=1e-14)
    odw = oracle.decode(qd, k, v, seqlens, window=5)
    for b in range(B):
        L = seqlens[b]
        full = oracle.attention(q[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L],
                                causal=True, window=5)
        np.testing.assert_allclose(odw[b, :, 0], full[0, :, L - 1], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- independent restatements

@pytest.mark.parametrize("causal,window,window_p4,hq,hkv", [
    (True, 0, False, 2, 2), (False, 0, False, 2, 2), (True, 3, False, 4, 2),
    (True, 2, True, 3, 1), (True, 0, False, 4, 4)])
def test_brute_force_agrees(causal, window, window_p4, hq, hkv):
    S, D = 7, 3
    q, k, v = _rand((1, hq, S, D), 27), _rand((1, hkv, S, D), 28), _rand((1, hkv, S, D), 29)
    o = oracle.attention(q, k, v, causal=causal, window=window, window_p4=window_p4)
    want = brute.attention(q[0].tolist(), k[0].tolist(), v[0].tolist(), causal=causal,
                           window=window, window_p4=window_p4)
    np.testing.assert_allclose(o[0], np.array(want), rtol=0, atol=1e-12)


def test_brute_force_agrees_on_a_cache_offset():
    """Query rows at positions q_pos0 + r against a longer key set."""
    Sq, Skv, D = 3, 8, 4
    q, k, v = _rand((1, 2, Sq, D), 30), _rand((1, 1, Skv, D), 31), _rand((1, 1, Skv, D), 32)
    o = oracle.attention(q, k, v, causal=True, q_pos0=[4], key_len=[7])
    want = brute.attention(q[0].tolist(), k[0].tolist(), v[0].tolist(), causal=True,
                           q_pos0=4, key_len=7)
    np.testing.assert_allclose(o[0], np.array(want), rtol=0, atol=1e-12)


def test_agrees_with_library_sdpa_in_float64():
    """torch.nn.functional.scaled_dot_product_attention (named on the textbook
    page, section "Эффективные реализации") computes the same definition."""
    import torch.nn.functional as F
    B, Hq, Hkv, S, D = 2, 4, 2, 45, 16
    q = torch.from_numpy(_rand((B, Hq, S, D), 33))
    k = torch.from_numpy(_rand((B, Hkv, S, D), 34))
    v = torch.from_numpy(_rand((B, Hkv, S, D), 35))
    kr, vr = k.repeat_interleave(2, dim=1), v.repeat_interleave(2, dim=1)
    ref = F.scaled_dot_product_attention(q, kr, vr, is_causal=True).numpy()
    np.testing.assert_allclose(oracle.attention(q, k, v, causal=True), ref, rtol=0, atol=1e-12)
    ref_nc = F.scaled_dot_product_attention(q, kr, vr, is_causal=False).numpy()
    np.testing.assert_allclose(oracle.attention(q, k, v, causal=False), ref_nc, rtol=0, atol=1e-12)
    W = 6
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    allowed = (j <= i) & (i - j < W)
    ref_w = F.scaled_dot_product_attention(q, kr, vr, attn_mask=allowed).numpy()
    np.testing.assert_allclose(oracle.attention(q, k, v, causal=True, window=W), ref_w,
                               rtol=0, atol=1e-12)
    sc = 0.3
    ref_s = F.scaled_dot_product_attention(q, kr, vr, is_causal=True, scale=sc).numpy()
    np.testing.assert_allclose(oracle.attention(q, k, v, causal=True, scale=sc), ref_s,
                               rtol=0, atol=1e-12)


def test_sampled_rows_match_full_rows():
    B, H, S, D = 1, 2, 70, 8
    q, k, v = _rand((B, H, S, D), 36), _rand((B, H, S, D), 37), _rand((B, H, S, D), 38)
    full = oracle.attention(q, k, v, causal=True, window=11)
    rows = [0, 10, 11, 69, 33]
    part = oracle.attention(q, k, v, causal=True, window=11, rows=rows)
    np.testing.assert_array_equal(part, full[:, :, rows])
