"""attn_decode_ring (decode over a rolling-buffer cache, through the C ABI):
position t of a sequence lives at cache row t % C.  Checked against the
float64 oracle on the logical sequence, including sequences that wrapped the
ring several times and 32-key blocks that straddle the wrap."""
import numpy as np
import pytest
import torch

import causal_head_self_gb300 as chs
import oracle
from causal_head_self_gb300 import build as _build
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    oracle.build()


def _ring_case(B, Hq, Hkv, C, Dh, lens, seed):
    """The logical q, K and V of each sequence and the ring buffers holding
    its last min(L, C) positions; rows never written hold large stale values
    so that reading one shows up."""
    gen = torch.Generator().manual_seed(seed)
    Lmax = max(lens)
    q = torch.randn((B, Hq, 1, Dh), generator=gen).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Lmax, Dh), generator=gen).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Lmax, Dh), generator=gen).to(torch.bfloat16)
    kr = torch.full((B, Hkv, C, Dh), 300.0).to(torch.bfloat16)
    vr = torch.full((B, Hkv, C, Dh), -300.0).to(torch.bfloat16)
    for b, L in enumerate(lens):
        t = torch.arange(max(0, L - C), L)
        kr[b, :, t % C] = k[b, :, t]
        vr[b, :, t % C] = v[b, :, t]
    return q, k, v, kr, vr, torch.tensor(lens, dtype=torch.int32)


def _run(q, kr, vr, sl, window):
    d = torch.device("cuda")
    o = chs.attn_decode_ring(q.to(d), kr.to(d), vr.to(d), sl.to(d), window=window)
    assert chs.attn_status() == chs.ATTN_OK
    return o.float().cpu().numpy()


# (B, Hq, Hkv, C, Dh, seqlens, window)
CASES = [
    (3, 8, 2, 1024, 128, [100, 1024, 3000], 0),        # not wrapped, full, wrapped twice
    (2, 32, 8, 4096, 128, [4096 * 3 + 17, 5000], 2048),  # window shorter than the ring
    (2, 4, 4, 300, 64, [299, 301], 0),                 # one head per CTA, Dh 64
    (2, 8, 4, 777, 128, [10000, 777 * 2], 500),        # ring not a multiple of a block
    (2, 8, 2, 640, 128, [639, 7001], 640),             # window == ring
    (1, 2, 2, 33, 128, [1000], 0),                     # a ring barely larger than a block
    (2, 8, 2, 500, 256, [1234, 499], 0),               # Dh 256: 16-key stages
    (2, 8, 2, 8192, 128, [8192 * 2 + 5, 9000], 0),     # wrapped, four 2048-key splits to merge
    (2, 4, 4, 8192, 128, [8192 * 2 + 5, 9000], 0),     # MHA (CUDA-core kernel), several splits
    (2, 4, 4, 500, 256, [1234, 499], 300),             # MHA at Dh 256 with a window
    # larger query-head groups: the tensor-core decode on the ring
    (2, 32, 1, 4096, 128, [4096 * 3 + 17, 5000], 2048), # MQA, window shorter than the ring
    (3, 16, 2, 1000, 128, [100, 1000, 3333], 0),       # not wrapped, full, wrapped
    (2, 8, 1, 777, 128, [10000, 777 * 2], 500),        # ring not a multiple of a tile
    (1, 32, 1, 33, 128, [1000], 0),                    # a ring smaller than one tile
    (2, 16, 2, 700, 256, [2345, 699], 0),              # Dh 256: 64-key tiles
    (2, 16, 1, 8192, 64, [8192 * 2 + 5, 9000], 0),     # Dh 64, several splits across the wrap
]


@pytest.mark.parametrize("B,Hq,Hkv,C,Dh,lens,window", CASES)
def test_ring_decode_against_oracle(B, Hq, Hkv, C, Dh, lens, window):
    q, k, v, kr, vr, sl = _ring_case(B, Hq, Hkv, C, Dh, lens, seed=C + Dh + window)
    got = _run(q, kr, vr, sl, window)
    w = window if window > 0 else C
    ref = oracle.attention(q, k, v, causal=True, window=w, key_len=np.array(lens),
                           q_pos0=np.array(lens) - 1)
    assert_close(got, ref, what=f"ring {(B, Hq, Hkv, C, Dh, lens, window)}")


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (32, 1)])   # CUDA-core, tensor-core, tensor-core
def test_unwrapped_ring_is_plain_decode_bitwise(Hq, Hkv):
    q, k, v, kr, vr, sl = _ring_case(3, Hq, Hkv, 2048, 128, [1, 700, 2048], seed=41)
    d = torch.device("cuda")
    a = chs.attn_decode(q.to(d), kr.to(d), vr.to(d), sl.to(d))
    b = chs.attn_decode_ring(q.to(d), kr.to(d), vr.to(d), sl.to(d))
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.equal(a, b)


def test_ring_rejects_a_window_wider_than_the_ring():
    q, k, v, kr, vr, sl = _ring_case(1, 2, 2, 64, 128, [100], seed=42)
    d = torch.device("cuda")
    with pytest.raises(chs.AttnError) as e:
        chs.attn_decode_ring(q.to(d), kr.to(d), vr.to(d), sl.to(d), window=65)
    assert e.value.code == chs.ATTN_ERR_INVALID_ARG
