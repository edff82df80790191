"""Failure detection without a GPU fault: the library's test hook withholds
one copy from a producer, so the kernels' bounded mbarrier waits run out
(about 2 s), every role leaves its loop, the CTA frees its tensor memory and
exits, and the device error word reports ATTN_ERR_TIMEOUT through
attn_status().  The next launch without the fault must be correct: the
context stays usable and no state (decode completion counters, barriers)
leaks into it."""
import numpy as np
import pytest
import torch

import causal_head_self_gb300 as chs
import oracle
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()
    yield
    chs.attn_debug_inject_fault(0)


def test_prefill_withheld_tile_times_out_then_recovers():
    d = torch.device("cuda")
    q, k, v = inputs.prefill_inputs(1, 4, 2, 600, 128, seed=21)
    qd, kd, vd = q.to(d), k.to(d), v.to(d)
    assert chs.attn_status() == chs.ATTN_OK
    chs.attn_debug_inject_fault(1)
    try:
        chs.attn_fwd(qd, kd, vd)
        assert chs.attn_status() == chs.ATTN_ERR_TIMEOUT
        assert chs.attn_status() == chs.ATTN_OK   # read and cleared
    finally:
        chs.attn_debug_inject_fault(0)
    o = chs.attn_fwd(qd, kd, vd)
    assert chs.attn_status() == chs.ATTN_OK
    assert_close(o.float().cpu().numpy(), oracle.attention(q, k, v, causal=True))


def test_decode_withheld_block_times_out_then_recovers():
    d = torch.device("cuda")
    # one query head per K/V head: the CUDA-core decode, whose hook is kind 2
    q, kc, vc, sl = inputs.decode_inputs(3, 8, 8, 3000, 128, 1000, 3000, seed=22)
    qd, kcd, vcd, sld = q.to(d), kc.to(d), vc.to(d), sl.to(d)
    assert chs.attn_status() == chs.ATTN_OK
    chs.attn_debug_inject_fault(2)
    try:
        chs.attn_decode(qd, kcd, vcd, sld)
        assert chs.attn_status() == chs.ATTN_ERR_TIMEOUT
    finally:
        chs.attn_debug_inject_fault(0)
    o = chs.attn_decode(qd, kcd, vcd, sld)
    assert chs.attn_status() == chs.ATTN_OK
    assert_close(o.float().cpu().numpy(), oracle.decode(q, kc, vc, sl))


def test_backward_withheld_block_times_out_then_recovers():
    d = torch.device("cuda")
    q, k, v = inputs.prefill_inputs(1, 4, 2, 300, 128, seed=23)
    dout = inputs.grad_inputs(q.shape, seed=23)
    qd, kd, vd, dd = q.to(d), k.to(d), v.to(d), dout.to(d)
    o, lse = chs.attn_fwd_lse(qd, kd, vd)
    assert chs.attn_status() == chs.ATTN_OK
    chs.attn_debug_inject_fault(4)
    try:
        chs.attn_bwd(qd, kd, vd, o, dd, lse)
        assert chs.attn_status() == chs.ATTN_ERR_TIMEOUT
    finally:
        chs.attn_debug_inject_fault(0)
    dq, dk, dv = chs.attn_bwd(qd, kd, vd, o, dd, lse)
    assert chs.attn_status() == chs.ATTN_OK
    rq, rk, rv = oracle.attention_bwd(q, k, v, dout, causal=True)
    for got, ref in zip((dq, dk, dv), (rq, rk, rv)):
        s = max(1.0, float(np.sqrt(np.mean(ref ** 2))))
        err = np.abs(got.float().cpu().numpy() - ref)
        assert np.all(err <= 2e-2 * s + 2.0 ** -7 * np.abs(ref))


def test_unknown_fault_kind_is_rejected():
    with pytest.raises(chs.AttnError):
        chs.attn_debug_inject_fault(7)
