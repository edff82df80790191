"""The textbook's worked example and exercise on the GPU path ("Механизм
внимания", sections "Численный пример" and "Вопросы и упражнения"): T = 3
tokens, head size d_h = 2, causal mask.  The kernels take head sizes 64, 128
or 256, so Q, K and V are padded with zero columns to 64 (zero columns add
nothing to a dot product, and the padded output columns are weighted sums of
zeros), and the scale is passed explicitly as 1/sqrt(2), the page's
1/sqrt(d_h).  The printed outputs are checked within the bf16 parity bar
(2e-2); the inputs are exact in bf16."""
import json
import math
import os

import numpy as np
import pytest
import torch

import causal_head_self_gb300 as chs
import oracle
from causal_head_self_gb300 import build as _build

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SCALE = 1.0 / math.sqrt(2.0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _padded(rows, dh=64):
    x = torch.zeros((1, 1, len(rows), dh), dtype=torch.bfloat16)
    x[0, 0, :, :len(rows[0])] = torch.tensor(rows, dtype=torch.bfloat16)
    return x.cuda()


def test_worked_example_on_the_gpu():
    g = _golden("worked_example_t3_dh2.json")
    q, k, v = _padded(g["Q"]), _padded(g["K"]), _padded(g["V"])
    o = chs.attn_fwd(q, k, v, causal=True, scale=SCALE)
    assert chs.attn_status() == chs.ATTN_OK
    got = o.float().cpu().numpy()[0, 0]
    np.testing.assert_allclose(got[:, :2], g["O_pytorch"], atol=2e-2)
    assert not got[:, 2:].any()


def test_exercise_one_on_the_gpu_and_as_a_decode_step():
    g = _golden("exercise1_t3_dh2.json")
    q, k, v = _padded(g["Q"]), _padded(g["K"]), _padded(g["V"])
    o = chs.attn_fwd(q, k, v, causal=True, scale=SCALE)
    assert chs.attn_status() == chs.ATTN_OK
    np.testing.assert_allclose(o.float().cpu().numpy()[0, 0, 2, :2], g["o_row2"], atol=2e-2)
    # the third token as a decode step against a cache of the three tokens
    sl = torch.tensor([3], dtype=torch.int32, device="cuda")
    od = chs.attn_decode(q[:, :, 2:3].contiguous(), k, v, sl, scale=SCALE)
    assert chs.attn_status() == chs.ATTN_OK
    np.testing.assert_allclose(od.float().cpu().numpy()[0, 0, 0, :2], g["o_row2"], atol=2e-2)


def test_worked_example_gradients_on_the_gpu():
    """The backward pass of the same example (dout of ones on the two real
    columns) against the float64 oracle's backward at the same padding."""
    g = _golden("worked_example_t3_dh2.json")
    q, k, v = _padded(g["Q"]), _padded(g["K"]), _padded(g["V"])
    dout = torch.zeros_like(q)
    dout[..., :2] = 1.0
    o, lse = chs.attn_fwd_lse(q, k, v, causal=True, scale=SCALE)
    dq, dk, dv = chs.attn_bwd(q, k, v, o, dout, lse, causal=True, scale=SCALE)
    assert chs.attn_status() == chs.ATTN_OK
    ref = oracle.attention_bwd(q.cpu(), k.cpu(), v.cpu(), dout.cpu(), causal=True, scale=SCALE)
    for got, want in zip((dq, dk, dv), ref):
        np.testing.assert_allclose(got.float().cpu().numpy(), want, atol=2e-2)
