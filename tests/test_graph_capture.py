"""The entry points inside CUDA graphs: captured once (after eager calls that
size the library's workspaces and set its kernels' attributes), replayed on
new inputs copied into the captured buffers, and compared with eager calls
bit for bit (every kernel is deterministic).  Captured together: a prefill, an
MHA decode step (CUDA-core kernel with its in-kernel merge), an MQA decode
step (tensor-core kernel and its dependent combine launch) and a forward +
backward pass.  A workspace that would have to grow inside a capture is
reported as ATTN_ERR_NO_MEMORY instead of calling cudaMalloc there."""
import pytest
import torch

import causal_head_self_gb300 as chs
from causal_head_self_gb300 import build as _build
from causal_head_self_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()


def _inputs(seed, d):
    pre = [x.to(d) for x in inputs.prefill_inputs(1, 8, 2, 700, 128, seed=seed)]
    dec = [x.to(d) for x in inputs.decode_inputs(4, 8, 8, 4096, 128, 1000, 4096, seed=seed)]
    mqa = [x.to(d) for x in inputs.decode_inputs(2, 32, 1, 6000, 128, 3000, 6000, seed=seed + 1)]
    dout = inputs.grad_inputs(pre[0].shape, seed=seed).to(d)
    return pre, dec, mqa, dout


def _step(pre, dec, mqa, dout, outs):
    q, k, v = pre
    o, od, om, ol, lse, dq, dk, dv = outs
    chs.attn_fwd(q, k, v, o)
    chs.attn_decode(*dec, od)
    chs.attn_decode(*mqa, om)
    chs.attn_fwd_lse(q, k, v, ol, lse)
    chs.attn_bwd(q, k, v, ol, dout, lse, dq, dk, dv)


def test_captured_step_replays_bit_for_bit():
    d = torch.device("cuda")
    pre, dec, mqa, dout = _inputs(1, d)
    q, k, v = pre
    outs = [torch.empty_like(q), torch.empty_like(dec[0]), torch.empty_like(mqa[0]),
            torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=d),
            torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    _step(pre, dec, mqa, dout, outs)           # sizes the workspaces, sets attributes
    torch.cuda.synchronize()
    assert chs.attn_status() == chs.ATTN_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(pre, dec, mqa, dout, outs)
    for seed in (2, 3):
        npre, ndec, nmqa, ndout = _inputs(seed, d)
        for dst, src in zip(pre + dec + mqa + [dout], npre + ndec + nmqa + [ndout]):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert chs.attn_status() == chs.ATTN_OK
        ref = [torch.empty_like(x) for x in outs]
        _step(npre, ndec, nmqa, ndout, ref)
        torch.cuda.synchronize()
        assert chs.attn_status() == chs.ATTN_OK
        for got, want in zip(outs, ref):
            assert torch.equal(got, want)


# the refused call launches nothing, so torch warns that the graph is empty
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_workspace_growth_inside_a_capture_is_refused():
    d = torch.device("cuda")
    # far more (batch, head, split) partials than any earlier call of the
    # suite needed (256 query heads on one K/V head, 64 sequences: about 17 MB)
    q, kc, vc, sl = (x.to(d) for x in inputs.decode_inputs(64, 256, 1, 4096, 128, 4000, 4096,
                                                            seed=9))
    o = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with pytest.raises(chs.AttnError) as e:
        with torch.cuda.graph(g):
            chs.attn_decode(q, kc, vc, sl, o)
    assert e.value.code == chs.ATTN_ERR_NO_MEMORY
    torch.cuda.synchronize()
    # outside the capture the same call grows the workspace and succeeds
    chs.attn_decode(q, kc, vc, sl, o)
    torch.cuda.synchronize()
    assert chs.attn_status() == chs.ATTN_OK


def test_binding_takes_the_current_stream():
    """A call without an explicit stream runs on torch's current stream: the
    default one, one set with torch.cuda.stream, and a graph's capture stream."""
    from causal_head_self_gb300 import _binding
    assert _binding._stream_handle(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert _binding._stream_handle(None) == s.cuda_stream
    g = torch.cuda.CUDAGraph()
    x = torch.zeros(1, device="cuda")
    with torch.cuda.graph(g):
        assert _binding._stream_handle(None) == torch.cuda.current_stream().cuda_stream
        x.add_(1)
    assert _binding._stream_handle(s) == s.cuda_stream
