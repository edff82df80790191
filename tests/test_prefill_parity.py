"""attn_fwd (tcgen05 prefill kernel, through the C ABI) against the float64
oracle on seeded inputs: every row at sizes the oracle finishes in seconds,
sampled rows at the full workload sizes, plus the invariants and edge cases."""
import numpy as np
import pytest
import torch

import causal_head_self_gb300 as chs
import oracle
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs
from parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()


def gpu_fwd(q, k, v, causal, window, scale=0.0):
    d = torch.device("cuda")
    o = chs.attn_fwd(q.to(d), k.to(d), v.to(d), causal=causal, window=window, scale=scale)
    assert chs.attn_status() == chs.ATTN_OK
    return o


# (B, Hq, Hkv, S, Dh, causal, window): several 128-row tiles, ragged tails,
# GQA / MQA groups, windows narrower and wider than a tile
SMALL = [
    (1, 2, 2, 128, 64, 1, 0),
    (1, 2, 2, 1, 128, 1, 0),
    (1, 2, 2, 2, 64, 1, 0),
    (1, 3, 3, 127, 128, 1, 0),
    (1, 2, 2, 129, 128, 1, 0),
    (2, 2, 2, 255, 64, 1, 0),
    (1, 2, 2, 257, 128, 1, 0),
    (1, 2, 2, 300, 128, 0, 0),
    (1, 2, 2, 513, 64, 0, 0),
    (2, 4, 4, 640, 128, 1, 0),
    (1, 8, 2, 384, 128, 1, 0),
    (2, 8, 1, 333, 64, 1, 0),
    (1, 4, 2, 700, 128, 1, 1),
    (1, 4, 2, 700, 128, 1, 17),
    (1, 4, 1, 700, 128, 1, 128),
    (1, 4, 2, 700, 64, 1, 200),
    (1, 2, 2, 1000, 128, 1, 300),
    (1, 2, 2, 1000, 128, 1, 256),
    (1, 2, 2, 1030, 128, 1, 1000),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,Dh,causal,window", SMALL)
def test_all_rows_small(B, Hq, Hkv, S, Dh, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=S + Dh + window)
    o = gpu_fwd(q, k, v, causal, window)
    ref = oracle.attention(q, k, v, causal=bool(causal), window=window)
    assert_close(o.float().cpu().numpy(), ref, what=f"{(B, Hq, Hkv, S, Dh, causal, window)}")


# Head size 128 runs on two kernels: up to 1536 keys per head the 64-key-tile
# kernel with two CTAs per SM (every Dh 128 case above), beyond that the
# ping-pong kernel.  Both sides of the switch, and ragged tails, windows and
# GQA / MQA groups on the ping-pong side.
SWITCH_128 = [
    (1, 2, 2, 1536, 128, 1, 0),    # the longest sequence on the 64-key kernel
    (1, 2, 2, 1537, 128, 1, 0),    # the shortest on the ping-pong kernel: a one-row tail
    (1, 3, 3, 1663, 128, 1, 0),
    (1, 2, 2, 1601, 128, 0, 0),
    (1, 4, 2, 1700, 128, 1, 17),
    (1, 4, 1, 1800, 128, 1, 300),
    (2, 8, 2, 1560, 128, 1, 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,Dh,causal,window", SWITCH_128)
def test_all_rows_both_head128_kernels(B, Hq, Hkv, S, Dh, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=S + window + 3)
    o = gpu_fwd(q, k, v, causal, window)
    ref = oracle.attention(q, k, v, causal=bool(causal), window=window)
    assert_close(o.float().cpu().numpy(), ref, what=f"{(B, Hq, Hkv, S, Dh, causal, window)}")


# More work items (256-row query blocks x heads) than SMs, so every CTA of the
# persistent kernel runs several in a row: the barrier phases, ring positions
# and tensor-memory accumulators carry from one item into the next.  Mixed
# item sizes, a last block whose second 128-row half is empty (S % 256 <= 128)
# or partly filled, GQA, windows, both head sizes.
PERSISTENT = [
    (3, 16, 4, 2900, 128, 1, 0),
    (2, 24, 8, 3000, 64, 1, 700),
    (2, 16, 16, 2000, 128, 0, 0),
    (1, 160, 160, 256, 128, 1, 0),
    (8, 40, 8, 130, 64, 1, 0),
    (4, 20, 5, 1500, 128, 1, 129),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,Dh,causal,window", PERSISTENT)
def test_all_rows_many_items_per_cta(B, Hq, Hkv, S, Dh, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=3 * S + Dh + window)
    o = gpu_fwd(q, k, v, causal, window)
    ref = oracle.attention(q, k, v, causal=bool(causal), window=window)
    assert_close(o.float().cpu().numpy(), ref, what=f"{(B, Hq, Hkv, S, Dh, causal, window)}")


def test_output_only_16_byte_aligned():
    """The output may start on any 16-byte boundary (the kernel then stores
    16 bytes at a time instead of 32); results are identical."""
    q, k, v = inputs.prefill_inputs(2, 4, 2, 300, 128, seed=12)
    d = torch.device("cuda")
    q, k, v = q.to(d), k.to(d), v.to(d)
    want = chs.attn_fwd(q, k, v)
    buf = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device=d)
    o = buf[8:].view(q.shape)
    assert o.data_ptr() % 32 == 16
    chs.attn_fwd(q, k, v, o)
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.equal(o, want)


def test_explicit_scale():
    q, k, v = inputs.prefill_inputs(1, 2, 2, 200, 128, seed=5)
    o = gpu_fwd(q, k, v, 1, 0, scale=0.05)
    assert_close(o.float().cpu().numpy(), oracle.attention(q, k, v, causal=True, scale=0.05))


def test_single_token_returns_v_exactly():
    q, k, v = inputs.prefill_inputs(2, 4, 2, 1, 128, seed=6)
    o = gpu_fwd(q, k, v, 1, 0).cpu()
    assert torch.equal(o, v.repeat_interleave(2, dim=1))


def test_identical_keys_give_prefix_mean():
    S = 300
    q, _, v = inputs.prefill_inputs(1, 1, 1, S, 128, seed=7)
    k = torch.zeros_like(q)
    k[:] = q[:, :, :1]
    o = gpu_fwd(q, k, v, 1, 0).float().cpu().numpy()[0, 0]
    vv = v.double().numpy()[0, 0]
    want = np.cumsum(vv, 0) / np.arange(1, S + 1)[:, None]
    assert_close(o, want)


def test_deterministic_and_causal():
    q, k, v = inputs.prefill_inputs(1, 4, 4, 777, 128, seed=8)
    o1 = gpu_fwd(q, k, v, 1, 0).cpu()
    o2 = gpu_fwd(q, k, v, 1, 0).cpu()
    assert torch.equal(o1, o2)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[:, :, -1] += 1
    k2[:, :, -1] += 1
    v2[:, :, -1] += 1
    o3 = gpu_fwd(q2, k2, v2, 1, 0).cpu()
    assert torch.equal(o1[:, :, :-1], o3[:, :, :-1])
    assert not torch.equal(o1[:, :, -1], o3[:, :, -1])


def test_gqa_is_mha_on_repeated_heads_bitwise():
    q, k, v = inputs.prefill_inputs(1, 8, 2, 400, 128, seed=9)
    a = gpu_fwd(q, k, v, 1, 64).cpu()
    b = gpu_fwd(q, k.repeat_interleave(4, 1).contiguous(), v.repeat_interleave(4, 1).contiguous(),
                1, 64).cpu()
    assert torch.equal(a, b)
    c = gpu_fwd(q, k[:, :1].contiguous(), v[:, :1].contiguous(), 1, 0).cpu()
    d = gpu_fwd(q, k[:, :1].expand(1, 8, 400, 128).contiguous(),
                v[:, :1].expand(1, 8, 400, 128).contiguous(), 1, 0).cpu()
    assert torch.equal(c, d)


def test_window_page_rule_is_window_plus_one():
    """The textbook's window 0 <= i-j <= W equals this API's window W + 1."""
    q, k, v = inputs.prefill_inputs(1, 2, 2, 500, 64, seed=10)
    o = gpu_fwd(q, k, v, 1, 33)
    assert_close(o.float().cpu().numpy(), oracle.attention(q, k, v, causal=True, window=32,
                                                           window_p4=True))


# ---------------------------------------------------------------- full workload sizes

def _full(name, rows_per_head, must):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_inputs(name)
    o = gpu_fwd(q, k, v, int(w["causal"]), w["window"])
    rows = sample_rows(w["S"], rows_per_head, seed=w["seed"], must=must)
    ref = oracle.attention(q, k, v, causal=w["causal"], window=w["window"], rows=rows)
    got = o[:, :, torch.from_numpy(rows).to(o.device)].float().cpu().numpy()
    assert_close(got, ref, what=name)


def test_workload_mha_s128_d64_all_rows():
    name = "prefill_mha_b1_h2_s128_d64"
    _full(name, 128, ())


def test_workload_mha_b2_s1024_all_rows():
    _full("prefill_mha_b2_h32_s1024_d128", 1024, ())


def test_workload_mha_s4096_sampled():
    _full("prefill_mha_b1_h32_s4096_d128", 64, (0, 127, 128, 255, 256, 4095))


def test_workload_mha_s4096_noncausal_sampled():
    _full("prefill_mha_b1_h32_s4096_d128_noncausal", 64, (0, 4095))


def test_workload_gqa_s32768_window_sampled():
    _full("prefill_gqa_b1_h32kv8_s32768_d128_w4096", 64, (0, 4095, 4096, 4097, 8191, 32767))


def test_empty_batch_or_sequence_is_a_no_op():
    d = torch.device("cuda")
    for shape_q, shape_kv in (((0, 4, 16, 128), (0, 2, 16, 128)), ((2, 4, 0, 128), (2, 2, 0, 128))):
        q = torch.empty(shape_q, dtype=torch.bfloat16, device=d)
        k = torch.empty(shape_kv, dtype=torch.bfloat16, device=d)
        o = chs.attn_fwd(q, k, k.clone())
        assert o.shape == q.shape
    assert chs.attn_status() == chs.ATTN_OK


def test_many_tiny_items_all_rows():
    """300 work items of a handful of rows each: every CTA runs two, on
    ragged single tiles."""
    q, k, v = inputs.prefill_inputs(50, 6, 2, 5, 128, seed=51)
    o = gpu_fwd(q, k, v, 1, 0)
    assert_close(o.float().cpu().numpy(), oracle.attention(q, k, v, causal=True))
