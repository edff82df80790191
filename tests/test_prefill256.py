"""attn_fwd and attn_fwd_chunk at head size 256 (the tcgen05 kernel with one
128-row sub-tile per work item and 64-key tiles), through the C ABI, against
the float64 oracle: every row at small sizes (ragged tails, GQA/MQA,
windows, non-causal, many items per CTA), sampled rows at the full workload
size, the chunked-prefill offsets, and the failure hook."""
import numpy as np
import pytest
import torch

import causal_head_self_gb300 as chs
import oracle
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs
from parity import assert_close, sample_rows

pytestmark = pytest.mark.gpu

DH = 256


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()
    yield
    chs.attn_debug_inject_fault(0)


def gpu_fwd(q, k, v, causal, window, scale=0.0):
    d = torch.device("cuda")
    o = chs.attn_fwd(q.to(d), k.to(d), v.to(d), causal=bool(causal), window=window, scale=scale)
    assert chs.attn_status() == chs.ATTN_OK
    return o


# (B, Hq, Hkv, S, causal, window): one and several 64-key tiles and 128-row
# items, ragged tails on both, GQA/MQA, windows narrower than a key tile,
# between a key tile and an item, and wider than an item
SMALL = [
    (1, 2, 2, 1, 1, 0),
    (1, 2, 2, 2, 1, 0),
    (1, 2, 2, 63, 1, 0),
    (1, 2, 2, 64, 1, 0),
    (1, 2, 2, 65, 1, 0),
    (1, 3, 3, 127, 1, 0),
    (1, 2, 2, 128, 1, 0),
    (1, 2, 2, 129, 1, 0),
    (2, 2, 2, 255, 1, 0),
    (1, 2, 2, 300, 0, 0),
    (1, 2, 1, 513, 0, 0),
    (2, 4, 4, 640, 1, 0),
    (1, 8, 2, 384, 1, 0),
    (2, 8, 1, 333, 1, 0),
    (1, 4, 2, 700, 1, 1),
    (1, 4, 2, 700, 1, 17),
    (1, 4, 1, 700, 1, 64),
    (1, 4, 2, 700, 1, 65),
    (1, 4, 2, 700, 1, 200),
    (1, 2, 2, 1030, 1, 1000),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,causal,window", SMALL)
def test_all_rows_small(B, Hq, Hkv, S, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, DH, seed=S + window + 7)
    o = gpu_fwd(q, k, v, causal, window)
    ref = oracle.attention(q, k, v, causal=bool(causal), window=window)
    assert_close(o.float().cpu().numpy(), ref, what=f"{(B, Hq, Hkv, S, causal, window)}")


# More 128-row items than SMs: every CTA runs several in a row, so barrier
# phases, the global key-tile counter, the two S buffers and O carry from one
# item into the next (items of different lengths, odd and even tile counts).
PERSISTENT = [
    (2, 16, 8, 1500, 1, 0),
    (1, 40, 8, 1000, 1, 300),
    (2, 16, 16, 700, 0, 0),
    (4, 40, 5, 130, 1, 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,causal,window", PERSISTENT)
def test_all_rows_many_items_per_cta(B, Hq, Hkv, S, causal, window):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, DH, seed=3 * S + window)
    o = gpu_fwd(q, k, v, causal, window)
    ref = oracle.attention(q, k, v, causal=bool(causal), window=window)
    assert_close(o.float().cpu().numpy(), ref, what=f"{(B, Hq, Hkv, S, causal, window)}")


def test_single_token_returns_v_exactly():
    q, k, v = inputs.prefill_inputs(2, 4, 2, 1, DH, seed=6)
    o = gpu_fwd(q, k, v, 1, 0).cpu()
    assert torch.equal(o, v.repeat_interleave(2, dim=1))


def test_explicit_scale_and_16_byte_aligned_output():
    q, k, v = inputs.prefill_inputs(1, 2, 2, 200, DH, seed=5)
    o = gpu_fwd(q, k, v, 1, 0, scale=0.03)
    assert_close(o.float().cpu().numpy(), oracle.attention(q, k, v, causal=True, scale=0.03))
    d = torch.device("cuda")
    qd, kd, vd = q.to(d), k.to(d), v.to(d)
    buf = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device=d)
    o2 = buf[8:].view(q.shape)
    assert o2.data_ptr() % 32 == 16
    chs.attn_fwd(qd, kd, vd, o2, scale=0.03)
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.equal(o2, o)


def test_deterministic_and_gqa_is_mha_on_repeated_heads():
    q, k, v = inputs.prefill_inputs(1, 8, 2, 400, DH, seed=9)
    a = gpu_fwd(q, k, v, 1, 64).cpu()
    assert torch.equal(a, gpu_fwd(q, k, v, 1, 64).cpu())
    b = gpu_fwd(q, k.repeat_interleave(4, 1).contiguous(), v.repeat_interleave(4, 1).contiguous(),
                1, 64).cpu()
    assert torch.equal(a, b)


def test_nan_canary_every_output_written():
    d = torch.device("cuda")
    q, k, v = inputs.prefill_inputs(2, 6, 3, 333, DH, seed=11)
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=d)
    chs.attn_fwd(q.to(d), k.to(d), v.to(d), o, window=100)
    assert chs.attn_status() == chs.ATTN_OK
    assert bool(torch.isfinite(o).all())


# ---------------------------------------------------------------- chunked prefill

# (B, Hq, Hkv, Sq, Tmax, start_pos, causal, window)
CHUNKS = [
    (1, 4, 2, 200, 1000, 300, 1, 0),
    (2, 4, 2, 128, 512, 256, 1, 0),
    (1, 4, 4, 130, 700, 555, 1, 100),
    (1, 2, 2, 1, 300, 299, 1, 0),
    (1, 4, 2, 150, 400, 200, 0, 0),
    (1, 2, 1, 65, 1200, 1000, 1, 333),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Tmax,start,causal,window", CHUNKS)
def test_chunk_all_rows(B, Hq, Hkv, Sq, Tmax, start, causal, window):
    q, kc, vc = inputs.prefill_inputs(B, Hq, Hkv, Tmax, DH, seed=start + Sq)
    q = q[:, :, :Sq].contiguous()
    # rows past the chunk are never read: poison them
    kc[:, :, start + Sq:] = float("nan")
    vc[:, :, start + Sq:] = float("nan")
    d = torch.device("cuda")
    o = chs.attn_fwd_chunk(q.to(d), kc.to(d), vc.to(d), start, causal=bool(causal), window=window)
    assert chs.attn_status() == chs.ATTN_OK
    ref = oracle.attention(q, kc[:, :, :start + Sq], vc[:, :, :start + Sq], causal=bool(causal),
                           window=window, q_pos0=[start] * B)
    assert_close(o.float().cpu().numpy(), ref, what=f"{(B, Hq, Hkv, Sq, Tmax, start)}")


def test_chunk_at_zero_equals_fwd_bitwise():
    q, k, v = inputs.prefill_inputs(1, 4, 2, 300, DH, seed=13)
    d = torch.device("cuda")
    a = chs.attn_fwd(q.to(d), k.to(d), v.to(d))
    b = chs.attn_fwd_chunk(q.to(d), k.to(d), v.to(d), 0)
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.equal(a, b)


# ---------------------------------------------------------------- full workload size

@pytest.mark.parametrize("name,must", [
    ("prefill_gqa_b1_h16kv8_s8192_d256", (0, 63, 64, 127, 128, 8191)),
    ("prefill_gqa_b1_h16kv8_s8192_d256_w4096", (0, 4095, 4096, 4097, 8191)),
])
def test_workload_sampled(name, must):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_inputs(name)
    o = gpu_fwd(q, k, v, int(w["causal"]), w["window"])
    rows = sample_rows(w["S"], 48, seed=w["seed"], must=must)
    ref = oracle.attention(q, k, v, causal=w["causal"], window=w["window"], rows=rows)
    got = o[:, :, torch.from_numpy(rows).to(o.device)].float().cpu().numpy()
    assert_close(got, ref, what=name)


# ---------------------------------------------------------------- failure hook

def test_withheld_tile_times_out_then_recovers():
    d = torch.device("cuda")
    q, k, v = inputs.prefill_inputs(1, 4, 2, 300, DH, seed=21)
    qd, kd, vd = q.to(d), k.to(d), v.to(d)
    assert chs.attn_status() == chs.ATTN_OK
    chs.attn_debug_inject_fault(1)
    try:
        chs.attn_fwd(qd, kd, vd)
        assert chs.attn_status() == chs.ATTN_ERR_TIMEOUT
    finally:
        chs.attn_debug_inject_fault(0)
    o = chs.attn_fwd(qd, kd, vd)
    assert chs.attn_status() == chs.ATTN_OK
    assert_close(o.float().cpu().numpy(), oracle.attention(q, k, v, causal=True))
