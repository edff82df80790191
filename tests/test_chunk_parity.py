"""attn_fwd_chunk (prefill of a chunk against a KV cache, through the C ABI)
against the float64 oracle with the chunk's queries at positions
start_pos .. start_pos + Sq - 1, plus the identities that tie it to attn_fwd
and attn_decode."""
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


def _chunk_inputs(B, Hq, Hkv, Sq, Tmax, Dh, seed):
    """q [B,Hq,Sq,Dh] and caches [B,Hkv,Tmax,Dh] (the chunk's own keys are
    whatever the cache holds at its rows)."""
    q, kc, vc = inputs.prefill_inputs(B, Hq, Hkv, Tmax, Dh, seed=seed)
    return q[:, :, :Sq].contiguous(), kc, vc


def _gpu_chunk(q, kc, vc, start, causal, window):
    d = torch.device("cuda")
    o = chs.attn_fwd_chunk(q.to(d), kc.to(d), vc.to(d), start, causal=bool(causal), window=window)
    assert chs.attn_status() == chs.ATTN_OK
    return o


def _oracle_chunk(q, kc, vc, start, causal, window, rows=None):
    Sq = q.shape[2]
    return oracle.attention(q, kc[:, :, :start + Sq], vc[:, :, :start + Sq], causal=bool(causal),
                            window=window, q_pos0=[start] * q.shape[0], rows=rows)


# (B, Hq, Hkv, Sq, Tmax, start_pos, Dh, causal, window)
CASES = [
    (1, 4, 2, 200, 1000, 300, 128, 1, 0),     # unaligned start, cache longer than needed
    (2, 8, 2, 256, 512, 256, 128, 1, 0),      # tile-aligned start
    (1, 4, 4, 130, 700, 555, 64, 1, 100),     # window, ragged chunk
    (1, 2, 2, 1, 300, 299, 128, 1, 0),        # one-token chunk
    (2, 4, 1, 300, 900, 0, 128, 1, 0),        # first chunk of a longer cache
    (1, 4, 2, 150, 400, 200, 128, 0, 0),      # non-causal: the whole cache plus chunk
    (1, 2, 2, 129, 1200, 1000, 128, 1, 333),  # window shorter than the cached prefix
    (3, 6, 3, 64, 3000, 2900, 64, 1, 0),      # short chunk after a long prefix
    # head size 128 past 1536 keys (the ping-pong kernel): ragged chunks
    (1, 4, 2, 129, 2500, 1700, 128, 1, 0),
    (1, 2, 2, 200, 2400, 2000, 128, 1, 500),
    (1, 4, 4, 100, 1536, 1436, 128, 1, 0),    # 1536 keys: the 64-key kernel
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Tmax,start,Dh,causal,window", CASES)
def test_chunk_all_rows(B, Hq, Hkv, Sq, Tmax, start, Dh, causal, window):
    q, kc, vc = _chunk_inputs(B, Hq, Hkv, Sq, Tmax, Dh, seed=start + Sq + Dh)
    o = _gpu_chunk(q, kc, vc, start, causal, window)
    assert_close(o.float().cpu().numpy(), _oracle_chunk(q, kc, vc, start, causal, window),
                 what=f"{(B, Hq, Hkv, Sq, Tmax, start, Dh, causal, window)}")


def test_chunk_many_items_sampled():
    """A 1024-token chunk after 2048 cached tokens, 32 query heads over 8 K/V
    heads: more work items than SMs; sampled rows against the oracle."""
    B, Hq, Hkv, Sq, Tmax, start, Dh = 2, 32, 8, 1024, 4096, 2048, 128
    q, kc, vc = _chunk_inputs(B, Hq, Hkv, Sq, Tmax, Dh, seed=31)
    o = _gpu_chunk(q, kc, vc, start, 1, 0)
    rows = sample_rows(Sq, 48, seed=31, must=(0, 127, 128, 255, 256, Sq - 1))
    ref = _oracle_chunk(q, kc, vc, start, 1, 0, rows=rows)
    got = o[:, :, torch.from_numpy(rows).to(o.device)].float().cpu().numpy()
    assert_close(got, ref, what="chunk 1024 after 2048")


def test_start_zero_full_cache_is_attn_fwd_bitwise():
    q, k, v = inputs.prefill_inputs(2, 8, 2, 700, 128, seed=32)
    d = torch.device("cuda")
    a = chs.attn_fwd(q.to(d), k.to(d), v.to(d))
    b = chs.attn_fwd_chunk(q.to(d), k.to(d), v.to(d), 0)
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.equal(a, b)


def test_chunks_reassemble_the_full_prefill():
    """Feeding a sequence in three chunks gives the rows of one full prefill
    (up to rounding: the tiles fall differently)."""
    S = 1024
    q, k, v = inputs.prefill_inputs(1, 8, 4, S, 128, seed=33)
    d = torch.device("cuda")
    qd, kd, vd = q.to(d), k.to(d), v.to(d)
    full = chs.attn_fwd(qd, kd, vd).float().cpu().numpy()
    parts, start = [], 0
    for n in (300, 500, 224):
        parts.append(chs.attn_fwd_chunk(qd[:, :, start:start + n].contiguous(), kd, vd, start)
                     .float().cpu().numpy())
        start += n
    assert chs.attn_status() == chs.ATTN_OK
    assert_close(np.concatenate(parts, axis=2), full, what="chunks vs full")


def test_one_token_chunk_matches_decode():
    B, Hq, Hkv, Tmax, Dh = 3, 8, 2, 2000, 128
    q, kc, vc, sl = inputs.decode_inputs(B, Hq, Hkv, Tmax, Dh, 1500, 1500, seed=34)
    d = torch.device("cuda")
    dec = chs.attn_decode(q.to(d), kc.to(d), vc.to(d), sl.to(d)).float().cpu().numpy()
    L = int(sl[0])
    ch = chs.attn_fwd_chunk(q.to(d), kc.to(d), vc.to(d), L - 1).float().cpu().numpy()
    assert chs.attn_status() == chs.ATTN_OK
    assert_close(ch, dec, what="one-token chunk vs decode")


def test_chunk_rejects_a_chunk_past_the_cache():
    q, kc, vc = _chunk_inputs(1, 2, 2, 100, 300, 64, seed=35)
    d = torch.device("cuda")
    with pytest.raises(chs.AttnError) as e:
        chs.attn_fwd_chunk(q.to(d), kc.to(d), vc.to(d), 201)
    assert e.value.code == chs.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("Dh", [64, 128])
def test_cache_rows_past_the_chunk_are_never_read(Dh):
    """Cache rows at or past start_pos + Sq hold NaN: the last key tile
    reaches past them (start_pos + Sq is not a multiple of the tile) but the
    output must not see them."""
    B, Hq, Hkv, Sq, Tmax, start = 2, 4, 2, 150, 900, 333
    q, kc, vc = _chunk_inputs(B, Hq, Hkv, Sq, Tmax, Dh, seed=36 + Dh)
    ref = _oracle_chunk(q, kc, vc, start, 1, 0)
    kc[:, :, start + Sq:] = float("nan")
    vc[:, :, start + Sq:] = float("nan")
    o = _gpu_chunk(q, kc, vc, start, 1, 0)
    assert_close(o.float().cpu().numpy(), ref, what="NaN past the chunk")
