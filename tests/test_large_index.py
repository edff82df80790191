"""Tensors past 2^31 elements and sequence positions near 2^31, through the
C ABI against the float64 oracle: 32-bit element offsets or positions would
wrap here.  A prefill whose q and o hold 2^31 elements each (sampled rows,
sliding window), decode over caches of 2^31 elements per K and V (every row
outside the visible window holds NaN, so a wrong address shows), and
rolling-buffer decode of sequences 2^31 - 1 tokens long."""
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


def test_prefill_with_q_and_o_of_2_31_elements():
    B, Hq, Hkv, S, Dh, W = 1, 64, 8, 262144, 128, 128
    d = torch.device("cuda")
    q = inputs.device_normal_bf16((B, Hq, S, Dh), 101, d)
    k = inputs.device_normal_bf16((B, Hkv, S, Dh), 102, d)
    v = inputs.device_normal_bf16((B, Hkv, S, Dh), 103, d)
    assert q.numel() == 2 ** 31
    o = chs.attn_fwd(q, k, v, window=W)
    assert chs.attn_status() == chs.ATTN_OK
    rows = sample_rows(S, 12, seed=7, must=(0, 1, W - 1, W, S // 2 - 1, S // 2, S - 2, S - 1))
    for h in (0, 31, 63):
        g = h // (Hq // Hkv)
        got, ref = [], []
        for i in rows:
            lo = max(0, int(i) - W + 1)
            # the row's visible keys only, all of them visible
            r = oracle.attention(q[:, h:h + 1, i:i + 1].cpu(), k[:, g:g + 1, lo:i + 1].cpu(),
                                 v[:, g:g + 1, lo:i + 1].cpu(), causal=False)
            ref.append(r[0, 0, 0])
            got.append(o[0, h, i].float().cpu().numpy())
        assert_close(np.array(got), np.array(ref), what=f"head {h}")
    del q, k, v, o


@pytest.mark.parametrize("Hq,Hkv,Dh", [(16384, 2048, 128), (8192, 1024, 256)])
def test_short_prefill_with_q_and_o_of_2_31_elements(Hq, Hkv, Dh):
    """The 64-key-tile kernel (head size 128 up to 1536 keys, and head size
    256): 1024 positions per head, so many heads that q and o hold 2^31
    elements; causal, sampled heads and rows (the last head's rows sit past
    2^31 elements)."""
    B, S = 1, 1024
    d = torch.device("cuda")
    q = inputs.device_normal_bf16((B, Hq, S, Dh), 111, d)
    k = inputs.device_normal_bf16((B, Hkv, S, Dh), 112, d)
    v = inputs.device_normal_bf16((B, Hkv, S, Dh), 113, d)
    assert q.numel() == 2 ** 31
    o = chs.attn_fwd(q, k, v)
    assert chs.attn_status() == chs.ATTN_OK
    rows = sample_rows(S, 8, seed=9, must=(0, 127, 128, S - 1))
    for h in (0, Hq // 2 - 1, Hq - 1):
        g = h // (Hq // Hkv)
        ref = oracle.attention(q[:, h:h + 1].cpu(), k[:, g:g + 1].cpu(), v[:, g:g + 1].cpu(),
                               causal=True, rows=rows)
        got = o[0, h, torch.from_numpy(rows).to(d)].float().cpu().numpy()
        assert_close(got, ref[0, 0], what=f"head {h}")
    del q, k, v, o


def _window_caches(B, Hkv, Tmax, Dh, lens, W, seed):
    """Caches of NaN except each sequence's last W positions, which hold
    i.i.d. N(0, 1) values; also those visible keys and values alone."""
    d = torch.device("cuda")
    kc = torch.full((B, Hkv, Tmax, Dh), float("nan"), dtype=torch.bfloat16, device=d)
    vc = torch.full((B, Hkv, Tmax, Dh), float("nan"), dtype=torch.bfloat16, device=d)
    q, kw, vw, _ = inputs.decode_inputs(B, 8 * Hkv, Hkv, W, Dh, 1, 1, seed)
    for b, L in enumerate(lens):
        kc[b, :, L - W:L] = kw[b].to(d)
        vc[b, :, L - W:L] = vw[b].to(d)
    return kc, vc, kw, vw


@pytest.mark.parametrize("Hq", [8, 64])   # CUDA-core kernel (MHA), tensor-core kernel
def test_decode_over_caches_of_2_31_elements(Hq):
    B, Hkv, Tmax, Dh, W = 2, 8, 2 ** 20, 128, 4096
    lens = [Tmax, Tmax - 777]
    kc, vc, kw, vw = _window_caches(B, Hkv, Tmax, Dh, lens, W, seed=Hq)
    assert kc.numel() == 2 ** 31
    gen = torch.Generator().manual_seed(Hq + 1)
    q = torch.randn((B, Hq, 1, Dh), generator=gen).to(torch.bfloat16)
    d = torch.device("cuda")
    sl = torch.tensor(lens, dtype=torch.int32, device=d)
    o = chs.attn_decode(q.to(d), kc, vc, sl, window=W)
    assert chs.attn_status() == chs.ATTN_OK
    ref = oracle.decode(q, kw, vw, np.full(B, W))
    assert_close(o.float().cpu().numpy(), ref, what=f"decode Hq={Hq}")
    del kc, vc


@pytest.mark.parametrize("Hq", [8, 64])   # CUDA-core kernel (MHA), tensor-core kernel
def test_ring_decode_at_positions_near_2_31(Hq):
    B, Hkv, C, Dh = 2, 8, 4096, 128
    lens = [2 ** 31 - 1, 2 ** 31 - 1 - 2500]
    q, kw, vw, _ = inputs.decode_inputs(B, Hq, Hkv, C, Dh, 1, 1, seed=Hq + 5)
    kr = torch.empty_like(kw)
    vr = torch.empty_like(vw)
    for b, L in enumerate(lens):
        rows = (torch.arange(L - C, L, dtype=torch.int64) % C)   # row of logical key j
        kr[b, :, rows] = kw[b]
        vr[b, :, rows] = vw[b]
    d = torch.device("cuda")
    sl = torch.tensor(lens, dtype=torch.int32, device=d)
    o = chs.attn_decode_ring(q.to(d), kr.to(d), vr.to(d), sl)
    assert chs.attn_status() == chs.ATTN_OK
    ref = oracle.decode(q, kw, vw, np.full(B, C))
    assert_close(o.float().cpu().numpy(), ref, what=f"ring Hq={Hq}")
