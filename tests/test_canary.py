"""NaN canaries: every output element is written.  The output buffer is
filled with NaN before each call; afterwards every element must be finite,
for ragged shapes of every entry point (a kernel that skipped a row, a
column block or a head would leave a NaN behind)."""
import pytest
import torch

import causal_head_self_gb300 as chs
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()


def _nan_like(x):
    return torch.full_like(x, float("nan"))


@pytest.mark.parametrize("B,Hq,Hkv,S,Dh,causal,window", [
    (2, 6, 3, 1, 128, 1, 0), (1, 4, 2, 129, 64, 1, 0), (3, 8, 1, 700, 128, 1, 200),
    (1, 2, 2, 513, 128, 0, 0), (2, 40, 8, 300, 128, 1, 0),
])
def test_prefill_writes_every_element(B, Hq, Hkv, S, Dh, causal, window):
    d = torch.device("cuda")
    q, k, v = (x.to(d) for x in inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=71 + S))
    o = chs.attn_fwd(q, k, v, _nan_like(q), causal=bool(causal), window=window)
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.isfinite(o).all()


def test_chunk_writes_every_element():
    d = torch.device("cuda")
    q, k, v = (x.to(d) for x in inputs.prefill_inputs(2, 8, 2, 1000, 128, seed=72))
    qc = q[:, :, :333].contiguous()
    o = chs.attn_fwd_chunk(qc, k, v, 555, _nan_like(qc))
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.isfinite(o).all()


@pytest.mark.parametrize("B,Hq,Hkv,Tmax,Dh", [
    (5, 8, 2, 2000, 128), (3, 12, 1, 900, 64), (2, 32, 1, 3000, 128), (2, 200, 1, 400, 128),
    (2, 8, 2, 500, 256),
])
def test_decode_writes_every_element(B, Hq, Hkv, Tmax, Dh):
    d = torch.device("cuda")
    q, kc, vc, sl = (x.to(d) for x in inputs.decode_inputs(B, Hq, Hkv, Tmax, Dh, 1, Tmax,
                                                           seed=73 + Tmax))
    o = chs.attn_decode(q, kc, vc, sl, _nan_like(q))
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.isfinite(o).all()
    o = chs.attn_decode_ring(q, kc, vc, sl, _nan_like(q))
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.isfinite(o).all()
    o = chs.attn_decode_noalloc(q, kc, vc, sl, _nan_like(q))
    assert chs.attn_status() == chs.ATTN_OK
    assert torch.isfinite(o).all()
