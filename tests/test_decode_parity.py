"""attn_decode (split-KV decode + combine kernels, through the C ABI) against
the float64 oracle on seeded inputs, edge cases, and the decode = last row of
prefill invariant."""
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


def gpu_decode(q, kc, vc, sl, window=0, scale=0.0, expect=chs.ATTN_OK):
    d = torch.device("cuda")
    o = chs.attn_decode(q.to(d), kc.to(d), vc.to(d), sl.to(d), window=window, scale=scale)
    assert chs.attn_status() == expect
    return o


# (B, Hq, Hkv, Tmax, Dh, lmin, lmax, window)
CASES = [
    (3, 8, 2, 1000, 128, 1, 1000, 0),
    (3, 8, 2, 1000, 128, 1, 1000, 300),
    (4, 8, 8, 700, 128, 100, 700, 0),     # MHA: one query head per K/V head
    (2, 4, 2, 3000, 128, 1500, 3000, 0),  # group of 2
    (2, 12, 1, 900, 128, 500, 900, 0),    # MQA, group of 12 (three CTAs per K/V head)
    (2, 3, 1, 513, 128, 1, 513, 64),      # group of 3
    (3, 8, 2, 2000, 64, 1, 2000, 0),
    (2, 16, 4, 5000, 64, 4000, 5000, 1000),
    (1, 32, 8, 20000, 128, 20000, 20000, 0),
    (3, 8, 2, 12000, 128, 9000, 12000, 0),  # several 2048-key splits per sequence
    (2, 8, 4, 12000, 64, 9000, 12000, 3000),
    # one query head per K/V head (the CUDA-core kernel): several splits,
    # windows, every head size
    (3, 4, 4, 12000, 128, 9000, 12000, 0),
    (2, 4, 4, 12000, 64, 1, 12000, 3000),
    (2, 4, 4, 9000, 256, 5000, 9000, 700),
    (5, 2, 2, 300, 128, 1, 300, 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,Tmax,Dh,lmin,lmax,window", CASES)
def test_decode_matches_oracle(B, Hq, Hkv, Tmax, Dh, lmin, lmax, window):
    q, kc, vc, sl = inputs.decode_inputs(B, Hq, Hkv, Tmax, Dh, lmin, lmax, seed=Tmax + Dh)
    if lmin == 1:
        sl[0] = 1   # a cache holding only the new token's own key
    o = gpu_decode(q, kc, vc, sl, window=window)
    ref = oracle.decode(q, kc, vc, sl, window=window)
    assert_close(o.float().cpu().numpy(), ref, what=str((B, Hq, Hkv, Tmax, Dh, window)))


def test_single_cached_key_returns_its_value():
    q, kc, vc, sl = inputs.decode_inputs(2, 8, 2, 64, 128, 1, 1, seed=3)
    o = gpu_decode(q, kc, vc, sl).cpu()
    assert torch.equal(o, vc[:, :, :1].repeat_interleave(4, dim=1))


def test_decode_equals_last_prefill_row():
    """"Prefill и decode": with the new token's key/value in the cache, the
    decode step reproduces the last row of a causal pass over the prefix."""
    S = 777
    q, k, v = inputs.prefill_inputs(2, 8, 2, S, 128, seed=11)
    full = chs.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True).float().cpu()
    for t in (0, 128, 400, S - 1):
        sl = torch.tensor([t + 1, t + 1], dtype=torch.int32)
        o = gpu_decode(q[:, :, t:t + 1].contiguous(), k, v, sl).float().cpu()
        assert_close(o.numpy(), full[:, :, t:t + 1].numpy(), max_abs=1.6e-2, mean_abs=2e-3)


def test_decode_is_deterministic():
    q, kc, vc, sl = inputs.decode_inputs(4, 8, 2, 4096, 128, 1000, 4096, seed=12)
    a = gpu_decode(q, kc, vc, sl).cpu()
    b = gpu_decode(q, kc, vc, sl).cpu()
    assert torch.equal(a, b)


def test_invalid_sequence_length_is_reported():
    q, kc, vc, sl = inputs.decode_inputs(3, 4, 4, 128, 64, 1, 128, seed=13)
    sl[1] = 0
    sl[2] = 129   # beyond Tmax
    o = gpu_decode(q, kc, vc, sl, expect=chs.ATTN_ERR_INVALID_ARG).cpu()
    assert torch.count_nonzero(o[1:]) == 0
    ref = oracle.decode(q[:1], kc[:1], vc[:1], sl[:1])
    assert_close(o[:1].float().numpy(), ref)
    assert chs.attn_status() == chs.ATTN_OK   # the latched code was cleared


def test_workload_decode_b16_all_rows():
    name = "decode_gqa_b16_h32kv8_t32768_d128"
    w = inputs.WORKLOADS[name]
    q, kc, vc, sl = inputs.workload_inputs(name)
    o = gpu_decode(q, kc, vc, sl, window=w["window"])
    ref = oracle.decode(q, kc, vc, sl, window=w["window"])
    assert_close(o.float().cpu().numpy(), ref, what=name)


def test_empty_batch_is_a_no_op():
    d = torch.device("cuda")
    q = torch.empty((0, 8, 1, 128), dtype=torch.bfloat16, device=d)
    kc = torch.empty((0, 2, 64, 128), dtype=torch.bfloat16, device=d)
    sl = torch.empty((0,), dtype=torch.int32, device=d)
    o = chs.attn_decode(q, kc, kc.clone(), sl)
    assert o.shape == q.shape
    assert chs.attn_status() == chs.ATTN_OK


def test_many_sequences_with_one_key_each():
    """B = 300 sequences of one cached key: the output is that key's value."""
    q, kc, vc, sl = inputs.decode_inputs(300, 4, 1, 32, 64, 1, 1, seed=52)
    o = gpu_decode(q, kc, vc, sl).cpu()
    assert torch.equal(o, vc[:, :1].repeat_interleave(4, dim=1)[:, :, :1])


@pytest.mark.parametrize("B,Hq,Hkv,Tmax,lmin,lmax,window", [
    (3, 8, 2, 3000, 1, 3000, 0),
    (2, 16, 1, 1000, 900, 1000, 300),   # MQA at Dh 256: the tensor-core path, 64-key tiles
    (2, 4, 4, 700, 1, 700, 0),
])
def test_head_size_256(B, Hq, Hkv, Tmax, lmin, lmax, window):
    """Dh = 256 (the Gemma head size): 16-key pipeline stages, a whole warp per key."""
    q, kc, vc, sl = inputs.decode_inputs(B, Hq, Hkv, Tmax, 256, lmin, lmax, seed=Tmax + 256)
    o = gpu_decode(q, kc, vc, sl, window=window)
    ref = oracle.decode(q, kc, vc, sl, window=window)
    assert_close(o.float().cpu().numpy(), ref, what=f"Dh 256 {(B, Hq, Hkv, Tmax, window)}")
