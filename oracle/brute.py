"""Pure-Python brute force of scaled dot-product attention, for tiny inputs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It exists to check the
C oracle by a second restatement that shares nothing with it: nested Python
lists, per-element loops, and the softmax taken straight from its formula
p_j = exp(s_j + M_j) / sum_k exp(s_k + M_k) without the max subtraction (fine
for the small scores of tiny inputs).  Masked keys contribute exp(-inf) = 0.

Definition: "Механизм внимания" (llm-arch-research.openidealab.com/textbook/attention),
section "Scaled dot-product attention"; head map g(h) = floor(h / (H/G)) from
section "Виды по числу голов K/V: MHA, GQA, MQA"; window from section
"Скользящее окно".
"""
from __future__ import annotations

import math


def attention(q, k, v, *, causal=True, window=0, window_p4=False, scale=None, q_pos0=0,
              key_len=None):
    """q: nested list [Hq][Sq][Dh]; k, v: [Hkv][Skv][Dh] (one sequence).
    Returns o as nested list [Hq][Sq][Dh]."""
    hq, hkv = len(q), len(k)
    sq, dh = len(q[0]), len(q[0][0])
    skv = len(k[0])
    if key_len is None:
        key_len = skv
    if scale is None:
        scale = 1.0 / math.sqrt(dh)
    out = []
    for h in range(hq):
        g = h // (hq // hkv)
        head = []
        for r in range(sq):
            i = q_pos0 + r
            weights = []
            for j in range(skv):
                allowed = j < key_len
                if causal and j > i:
                    allowed = False
                if window > 0:
                    if window_p4 and i - j > window:
                        allowed = False
                    if not window_p4 and i - j >= window:
                        allowed = False
                if allowed:
                    s = 0.0
                    for d in range(dh):
                        s += q[h][r][d] * k[g][j][d]
                    weights.append(math.exp(s * scale))
                else:
                    weights.append(0.0)
            total = 0.0
            for w in weights:
                total += w
            row = []
            for d in range(dh):
                acc = 0.0
                for j in range(skv):
                    acc += (weights[j] / total) * v[g][j][d]
                row.append(acc)
            head.append(row)
        out.append(head)
    return out
