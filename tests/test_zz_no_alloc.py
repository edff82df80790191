"""attn_decode_noalloc: the decode step for callers that must not allocate
device memory (a serving runtime that has reserved the device memory for its
own KV-cache pool, or a process under a fixed device-memory budget).  Its
scratch is a fixed device array inside the library instead of a cudaMalloc'd
workspace, so its results are checked against attn_decode, through the C ABI,
on two calls in a row (the second call finds the first call's contents in the
shared array).  This file is collected last on purpose."""
import ctypes

import pytest
import torch

import causal_head_self_gb300 as chs
from causal_head_self_gb300 import _binding
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()


# (B, Hq, Hkv, Tmax, Dh, lmin, lmax, window): several splits per sequence
CASES = [
    (4, 32, 8, 4096, 128, 1000, 4096, 0),
    (3, 8, 2, 5000, 64, 1, 5000, 3000),
    (4, 32, 1, 9000, 128, 3000, 9000, 0),    # MQA: the tensor-core path and its combine
    (3, 16, 2, 6000, 256, 2000, 6000, 0),    # group of 8 at Dh 256: tensor cores, 64-key tiles
    (4, 8, 8, 9000, 128, 3000, 9000, 0),     # MHA: the CUDA-core kernel, its counters in the array
    (3, 4, 4, 5000, 64, 1, 5000, 2000),      # MHA at Dh 64 with a window
]


@pytest.mark.parametrize("B,Hq,Hkv,Tmax,Dh,lmin,lmax,window", CASES)
def test_noalloc_matches_decode_on_two_calls(B, Hq, Hkv, Tmax, Dh, lmin, lmax, window):
    d = torch.device("cuda")
    q, kc, vc, sl = (x.to(d) for x in inputs.decode_inputs(B, Hq, Hkv, Tmax, Dh, lmin, lmax,
                                                             seed=77 + Dh))
    ref = chs.attn_decode(q, kc, vc, sl, window=window)
    assert chs.attn_status() == chs.ATTN_OK
    ref = ref.float().cpu().numpy()
    for _ in range(2):
        o = chs.attn_decode_noalloc(q, kc, vc, sl, window=window)
        assert chs.attn_status() == chs.ATTN_OK
        assert_close(o.float().cpu().numpy(), ref, what="noalloc vs decode")
        # the same kernels and split plan as attn_decode: the same bits
        assert (o.float().cpu().numpy() == ref).all()


SCRATCH_BYTES = 16 << 20   # the fixed array's size, as the header states


def test_noalloc_rejects_a_call_beyond_its_scratch():
    """A call whose split partials cannot fit the 16 MiB scratch is refused
    before anything is launched, so its pointers are never dereferenced.
    The shape is chosen so that even a single split per sequence needs more
    than the scratch (the header's formula: B*Hq*nsplit*(Dh+2)*4 bytes of
    partials, nsplit >= 1), whatever split plan the library picks; the
    assertion below checks that on the host before the call is made."""
    B, Hq, Hkv, Tmax, Dh = 2048, 32, 8, 64, 128
    min_partials = B * Hq * 1 * (Dh + 2) * 4
    assert min_partials > SCRATCH_BYTES, "the refusal must not depend on the split plan"
    lib = _binding.load()
    torch.cuda.init()
    big = 1 << 40
    rc = lib.attn_decode_noalloc(0x10000, big, 2 * big, 3 * big, 4 * big, B, Hq, Hkv, Tmax, Dh,
                                 0, 0.0, None)
    assert rc == chs.ATTN_ERR_SCRATCH_LIMIT
    assert chs.error_string(rc) == "ATTN_ERR_SCRATCH_LIMIT"
