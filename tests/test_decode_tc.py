"""The tensor-core decode path (taken by attn_decode when Hq / Hkv >= 2:
several query heads share each cached K/V row) against the float64 oracle,
and against the CUDA-core path on the same step with the K/V heads repeated."""
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


def _gpu(q, kc, vc, sl, window=0, expect=chs.ATTN_OK):
    d = torch.device("cuda")
    o = chs.attn_decode(q.to(d), kc.to(d), vc.to(d), sl.to(d), window=window)
    assert chs.attn_status() == expect
    return o


# (B, Hq, Hkv, Tmax, Dh, lmin, lmax, window)
CASES = [
    (4, 32, 1, 5000, 128, 1, 5000, 0),        # MQA, lengths from 1 key up
    (2, 16, 2, 3000, 64, 200, 3000, 700),     # group of 8, Dh 64, window
    (1, 200, 1, 1000, 128, 1000, 1000, 0),    # 200 heads on one K/V head: two row blocks
    (3, 64, 4, 300, 128, 1, 300, 0),          # group of 16, short caches
    (2, 32, 1, 20000, 128, 12000, 20000, 0),  # many splits per sequence
    (2, 40, 5, 777, 128, 129, 777, 128),      # window of exactly one tile
    # head size 256: 64-key tiles
    (4, 8, 1, 5000, 256, 1, 5000, 0),         # 8 heads on one K/V head, lengths from 1 key up
    (2, 16, 2, 3000, 256, 200, 3000, 700),    # group of 8, window
    (1, 200, 1, 1000, 256, 1000, 1000, 0),    # two row blocks
    (2, 32, 1, 20000, 256, 12000, 20000, 0),  # many splits per sequence
    (2, 40, 5, 777, 256, 65, 777, 64),        # window of exactly one 64-key tile
    # small groups: 2, 3 and 4 query heads per K/V head
    (3, 8, 4, 5000, 64, 1, 5000, 0),
    (2, 12, 4, 3000, 256, 1, 3000, 500),
    (4, 32, 8, 9000, 128, 2000, 9000, 0),
    (3, 6, 3, 4100, 128, 1, 4100, 1000),
]


@pytest.mark.parametrize("B,Hq,Hkv,Tmax,Dh,lmin,lmax,window", CASES)
def test_tc_decode_matches_oracle(B, Hq, Hkv, Tmax, Dh, lmin, lmax, window):
    q, kc, vc, sl = inputs.decode_inputs(B, Hq, Hkv, Tmax, Dh, lmin, lmax, seed=Tmax + Hq)
    o = _gpu(q, kc, vc, sl, window)
    ref = oracle.decode(q, kc, vc, sl, window=window)
    assert_close(o.float().cpu().numpy(), ref, what=str((B, Hq, Hkv, Tmax, Dh, window)))


def test_tc_path_agrees_with_the_cuda_core_path():
    """The same step with each K/V head repeated for its query heads (one
    query head per K/V head) runs on the CUDA-core kernel."""
    q, kc, vc, sl = inputs.decode_inputs(3, 16, 1, 2000, 128, 700, 2000, seed=61)
    a = _gpu(q, kc, vc, sl).float().cpu().numpy()
    b = _gpu(q, kc.expand(3, 16, 2000, 128).contiguous(),
             vc.expand(3, 16, 2000, 128).contiguous(), sl).float().cpu().numpy()
    assert_close(a, b, what="tensor-core vs CUDA-core decode")


@pytest.mark.parametrize("Dh", [128, 256])
def test_tc_cache_rows_past_the_length_are_not_read(Dh):
    """NaN in every cache row at or past seqlens[b] must not reach the output."""
    q, kc, vc, sl = inputs.decode_inputs(2, 32, 1, 1000, Dh, 130, 700, seed=62)
    ref = oracle.decode(q, kc, vc, sl)   # (the oracle touches every row, weighting hidden ones 0)
    for b, L in enumerate(sl.tolist()):
        kc[b, :, L:] = float("nan")
        vc[b, :, L:] = float("nan")
    o = _gpu(q, kc, vc, sl)
    assert_close(o.float().cpu().numpy(), ref)


def test_tc_invalid_length_is_reported():
    q, kc, vc, sl = inputs.decode_inputs(2, 16, 1, 256, 128, 1, 256, seed=63)
    sl[1] = 257
    o = _gpu(q, kc, vc, sl, expect=chs.ATTN_ERR_INVALID_ARG).float().cpu()
    assert torch.all(o[1] == 0)
    assert_close(o[:1].numpy(), oracle.decode(q[:1], kc[:1], vc[:1], sl[:1]))


def test_tc_withheld_tile_times_out_then_recovers():
    q, kc, vc, sl = inputs.decode_inputs(2, 32, 1, 600, 128, 300, 600, seed=64)
    chs.attn_debug_inject_fault(3)
    try:
        _gpu(q, kc, vc, sl, expect=chs.ATTN_ERR_TIMEOUT)
    finally:
        chs.attn_debug_inject_fault(0)
    o = _gpu(q, kc, vc, sl)
    assert_close(o.float().cpu().numpy(), oracle.decode(q, kc, vc, sl))
