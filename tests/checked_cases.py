"""Parity cases run against the range-checked build of the library (started
by tests/test_checked_build.py in a process of its own with
CHS_ATTN_CHECK=1): every kernel family, ragged tails, windows, rings that
wrap, chunks and the backward pass.  Exits non-zero on the first failure."""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import causal_head_self_gb300 as chs  # noqa: E402
import oracle  # noqa: E402
from causal_head_self_gb300 import inputs  # noqa: E402
from parity import assert_close  # noqa: E402


def status_ok(what):
    rc = chs.attn_status()
    assert rc == chs.ATTN_OK, f"{what}: {chs.error_string(rc)}"


def prefill_cases(d):
    for B, Hq, Hkv, S, Dh, causal, window in [(1, 4, 2, 300, 128, 1, 0), (2, 2, 1, 257, 64, 1, 77),
                                              (1, 2, 2, 200, 128, 0, 0), (1, 4, 2, 333, 256, 1, 0),
                                              (1, 2, 1, 200, 256, 1, 65)]:
        q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=S + Dh)
        o = chs.attn_fwd(q.to(d), k.to(d), v.to(d), causal=bool(causal), window=window)
        status_ok("prefill")
        ref = oracle.attention(q, k, v, causal=bool(causal), window=window)
        assert_close(o.float().cpu().numpy(), ref, what=f"prefill {(B, Hq, Hkv, S, Dh, causal, window)}")


def chunk_cases(d):
    for B, Hq, Hkv, Tmax, Sq, start, Dh in [(1, 4, 2, 700, 150, 500, 128), (1, 2, 1, 500, 100, 300, 256)]:
        q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Tmax, Dh, seed=Sq + start)
        qc = q[:, :, start:start + Sq].contiguous()
        o = chs.attn_fwd_chunk(qc.to(d), k.to(d), v.to(d), start)
        status_ok("chunk")
        ref = oracle.attention(qc, k[:, :, :start + Sq], v[:, :, :start + Sq], causal=True,
                               q_pos0=np.full(B, start))
        assert_close(o.float().cpu().numpy(), ref, what=f"chunk {(Hq, Hkv, Sq, start, Dh)}")


def decode_cases(d):
    for B, Hq, Hkv, Tmax, Dh, window in [(3, 8, 2, 3000, 128, 0), (2, 32, 1, 5000, 128, 700),
                                         (2, 8, 2, 1200, 256, 0), (2, 16, 2, 900, 256, 300),
                                         (2, 8, 2, 2000, 64, 0),
                                         # one query head per K/V head: the CUDA-core kernel
                                         (3, 4, 4, 9000, 128, 0), (2, 4, 4, 1200, 256, 300),
                                         (2, 4, 4, 5000, 64, 700)]:
        q, kc, vc, sl = inputs.decode_inputs(B, Hq, Hkv, Tmax, Dh, 1, Tmax, seed=Tmax + Dh)
        o = chs.attn_decode(q.to(d), kc.to(d), vc.to(d), sl.to(d), window=window)
        status_ok("decode")
        ref = oracle.decode(q, kc, vc, sl, window=window)
        assert_close(o.float().cpu().numpy(), ref, what=f"decode {(B, Hq, Hkv, Tmax, Dh, window)}")


def ring_cases(d):
    for B, Hq, Hkv, C, Dh, lens in [(2, 8, 2, 777, 128, [10000, 1554]), (2, 32, 1, 700, 128, [5000, 699]),
                                    (2, 16, 2, 500, 256, [2345, 499]),
                                    (2, 4, 4, 777, 128, [10000, 1554]), (2, 4, 4, 500, 256, [2345, 499])]:
        gen = torch.Generator().manual_seed(C + Hq)
        Lmax = max(lens)
        q = torch.randn((B, Hq, 1, Dh), generator=gen).to(torch.bfloat16)
        k = torch.randn((B, Hkv, Lmax, Dh), generator=gen).to(torch.bfloat16)
        v = torch.randn((B, Hkv, Lmax, Dh), generator=gen).to(torch.bfloat16)
        kr = torch.zeros((B, Hkv, C, Dh), dtype=torch.bfloat16)
        vr = torch.zeros((B, Hkv, C, Dh), dtype=torch.bfloat16)
        for b, L in enumerate(lens):
            t = torch.arange(max(0, L - C), L)
            kr[b, :, t % C] = k[b, :, t]
            vr[b, :, t % C] = v[b, :, t]
        sl = torch.tensor(lens, dtype=torch.int32)
        o = chs.attn_decode_ring(q.to(d), kr.to(d), vr.to(d), sl.to(d))
        status_ok("ring")
        ref = oracle.attention(q, k, v, causal=True, window=C, key_len=np.array(lens),
                               q_pos0=np.array(lens) - 1)
        assert_close(o.float().cpu().numpy(), ref, what=f"ring {(B, Hq, Hkv, C, Dh)}")


def backward_cases(d):
    for B, Hq, Hkv, S, Dh, window in [(1, 4, 2, 300, 128, 0), (1, 2, 1, 257, 64, 100),
                                      (1, 4, 2, 300, 256, 0), (1, 2, 1, 257, 256, 100)]:
        q, k, v = inputs.prefill_inputs(B, Hq, Hkv, S, Dh, seed=S)
        dout = inputs.grad_inputs(q.shape, seed=S)
        qd, kd, vd, dd = q.to(d), k.to(d), v.to(d), dout.to(d)
        o, lse = chs.attn_fwd_lse(qd, kd, vd, window=window)
        dq, dk, dv = chs.attn_bwd(qd, kd, vd, o, dd, lse, window=window)
        status_ok("backward")
        rq, rk, rv = oracle.attention_bwd(q, k, v, dout, causal=True, window=window)
        for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
            g = got.float().cpu().numpy()
            err = np.abs(g - ref)
            assert np.all(err <= 2e-2 + 2.0 ** -8 * np.abs(ref)), f"backward {name}"


def main():
    assert chs._binding.LIB_PATH.endswith("_check.so"), chs._binding.LIB_PATH
    oracle.build()
    d = torch.device("cuda")
    for fn in (prefill_cases, chunk_cases, decode_cases, ring_cases, backward_cases):
        fn(d)
        print(fn.__name__, "ok", flush=True)


if __name__ == "__main__":
    main()
