"""Seeded synthetic inputs, shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it only draws numbers.  Every
tensor is i.i.d. N(0, 1) (the unit-variance query/key assumption of
"Механизм внимания", section "Почему делить на корень из d_h"), drawn in
float32 from one ``torch.Generator('cpu')`` seeded per workload and rounded
to bfloat16, in the fixed order Q, K, V, then (for a decode step) the
per-sequence cache lengths.  The same host tensors feed both sides.
"""
from __future__ import annotations

import torch

# The workloads, named by what they are.  ``seed`` fixes every number drawn.
WORKLOADS = {
    # causal MHA core attention, the smallest case (every row checked)
    "prefill_mha_b1_h2_s128_d64": dict(kind="prefill", B=1, Hq=2, Hkv=2, S=128, Dh=64,
                                       causal=True, window=0, seed=0),
    # causal MHA prefill, hidden 4096 = 32 heads x 128
    "prefill_mha_b2_h32_s1024_d128": dict(kind="prefill", B=2, Hq=32, Hkv=32, S=1024, Dh=128,
                                          causal=True, window=0, seed=1),
    # causal MHA prefill at 4096 tokens, and its non-causal counterpart
    "prefill_mha_b1_h32_s4096_d128": dict(kind="prefill", B=1, Hq=32, Hkv=32, S=4096, Dh=128,
                                          causal=True, window=0, seed=2),
    "prefill_mha_b1_h32_s4096_d128_noncausal": dict(kind="prefill", B=1, Hq=32, Hkv=32, S=4096,
                                                    Dh=128, causal=False, window=0, seed=2),
    # causal GQA prefill (32 query heads over 8 K/V heads) with a 4096-key sliding window
    "prefill_gqa_b1_h32kv8_s32768_d128_w4096": dict(kind="prefill", B=1, Hq=32, Hkv=8, S=32768,
                                                    Dh=128, causal=True, window=4096, seed=3),
    # causal GQA prefill at head size 256 (16 query heads over 8 K/V heads),
    # without and with a 4096-key sliding window
    "prefill_gqa_b1_h16kv8_s8192_d256": dict(kind="prefill", B=1, Hq=16, Hkv=8, S=8192, Dh=256,
                                             causal=True, window=0, seed=6),
    "prefill_gqa_b1_h16kv8_s8192_d256_w4096": dict(kind="prefill", B=1, Hq=16, Hkv=8, S=8192,
                                                   Dh=256, causal=True, window=4096, seed=6),
    # the backward pass of causal MHA at 4096 tokens (and of the GQA prefill)
    "backward_mha_b1_h32_s4096_d128": dict(kind="backward", B=1, Hq=32, Hkv=32, S=4096, Dh=128,
                                           causal=True, window=0, seed=2),
    "backward_gqa_b2_h32kv8_s2048_d128": dict(kind="backward", B=2, Hq=32, Hkv=8, S=2048,
                                              Dh=128, causal=True, window=0, seed=7),
    # the backward pass at head size 256 (the causal GQA prefill at Dh=256)
    "backward_gqa_b1_h16kv8_s8192_d256": dict(kind="backward", B=1, Hq=16, Hkv=8, S=8192, Dh=256,
                                              causal=True, window=0, seed=6),
    # the Dh=256 backward on 4 query heads over 2 K/V heads at S=4096 (a profiler-sized case)
    "backward_gqa_b1_h4kv2_s4096_d256": dict(kind="backward", B=1, Hq=4, Hkv=2, S=4096, Dh=256,
                                             causal=True, window=0, seed=6),
    # the S=4096 backward on 8 heads (a profiler-sized case)
    "backward_mha_b1_h8_s4096_d128": dict(kind="backward", B=1, Hq=8, Hkv=8, S=4096, Dh=128,
                                          causal=True, window=0, seed=2),
    # chunked prefill: a 1024-token chunk after 3072 cached tokens (cache of 4096 rows)
    "chunk_gqa_b2_h32kv8_c1024_at3072_d128": dict(kind="chunk", B=2, Hq=32, Hkv=8, Sq=1024,
                                                  Tmax=4096, start=3072, Dh=128, causal=True,
                                                  window=0, seed=8),
    # rolling-buffer decode: a 4096-row ring per (sequence, K/V head) holding the
    # last 4096 of 16384..32768 positions, window 4096
    "ring_decode_gqa_b16_h32kv8_c4096_d128": dict(kind="ring", B=16, Hq=32, Hkv=8, Tmax=4096,
                                                  Dh=128, lmin=16384, lmax=32768, window=4096,
                                                  seed=9),
    # the same rolling-buffer decode with 32 query heads on one K/V head (tensor cores)
    "ring_decode_mqa_b16_h32kv1_c4096_d128": dict(kind="ring", B=16, Hq=32, Hkv=1, Tmax=4096,
                                                  Dh=128, lmin=16384, lmax=32768, window=4096,
                                                  seed=13),
    # MQA decode: 32 query heads on one K/V head (the tensor-core decode path)
    "decode_mqa_b16_h32kv1_t32768_d128": dict(kind="decode", B=16, Hq=32, Hkv=1, Tmax=32768,
                                              Dh=128, lmin=16384, lmax=32768, window=0, seed=10),
    # MQA decode at head size 256: 8 query heads on 1 K/V head (the Gemma-2B shape)
    "decode_mqa_b16_h8kv1_t32768_d256": dict(kind="decode", B=16, Hq=8, Hkv=1, Tmax=32768,
                                             Dh=256, lmin=16384, lmax=32768, window=0, seed=12),
    # one decode step for 16 sequences against caches of 16384..32768 keys
    "decode_gqa_b16_h32kv8_t32768_d128": dict(kind="decode", B=16, Hq=32, Hkv=8, Tmax=32768,
                                              Dh=128, lmin=16384, lmax=32768, window=0, seed=4),
    # the same decode step at head size 64
    "decode_gqa_b16_h32kv8_t32768_d64": dict(kind="decode", B=16, Hq=32, Hkv=8, Tmax=32768,
                                             Dh=64, lmin=16384, lmax=32768, window=0, seed=14),
    # the same decode step for 4 sequences (0.5 GB of cache: a profiler-sized case)
    "decode_gqa_b4_h32kv8_t32768_d128": dict(kind="decode", B=4, Hq=32, Hkv=8, Tmax=32768,
                                             Dh=128, lmin=16384, lmax=32768, window=0, seed=5),
}


def _randn_bf16(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(B, Hq, Hkv, S, Dh, seed):
    """q [B,Hq,S,Dh], k and v [B,Hkv,S,Dh], bf16 on the host."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    q = _randn_bf16((B, Hq, S, Dh), gen)
    k = _randn_bf16((B, Hkv, S, Dh), gen)
    v = _randn_bf16((B, Hkv, S, Dh), gen)
    return q, k, v


def device_normal_bf16(shape, seed, device):
    """i.i.d. N(0, 1) drawn on `device` by torch's generator, rounded to bf16:
    for tensors too large to draw on the host.  Drawn one slice of the first
    two axes at a time, so no full-size float32 copy is ever held."""
    gen = torch.Generator(device=device).manual_seed(int(seed))
    out = torch.empty(tuple(shape), dtype=torch.bfloat16, device=device)
    for i in range(shape[0]):
        for j in range(shape[1]):
            out[i, j] = torch.randn(tuple(shape[2:]), generator=gen, device=device,
                                    dtype=torch.float32).to(torch.bfloat16)
    return out


def grad_inputs(shape, seed):
    """An upstream gradient dL/do of the given shape: i.i.d. N(0, 1), bf16 on
    the host (its own generator, so adding it changes no other draw)."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed) + 7919)
    return _randn_bf16(tuple(shape), gen)


def decode_inputs(B, Hq, Hkv, Tmax, Dh, lmin, lmax, seed):
    """q [B,Hq,1,Dh], kcache and vcache [B,Hkv,Tmax,Dh] (bf16), and the
    per-sequence key counts seqlens [B] (int32, uniform in [lmin, lmax])."""
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    q = _randn_bf16((B, Hq, 1, Dh), gen)
    kc = _randn_bf16((B, Hkv, Tmax, Dh), gen)
    vc = _randn_bf16((B, Hkv, Tmax, Dh), gen)
    seqlens = torch.randint(int(lmin), int(lmax) + 1, (B,), generator=gen, dtype=torch.int64)
    return q, kc, vc, seqlens.to(torch.int32)


def workload_inputs(name):
    """The inputs of a named workload (see WORKLOADS)."""
    w = WORKLOADS[name]
    if w["kind"] == "prefill":
        return prefill_inputs(w["B"], w["Hq"], w["Hkv"], w["S"], w["Dh"], w["seed"])
    if w["kind"] == "backward":
        q, k, v = prefill_inputs(w["B"], w["Hq"], w["Hkv"], w["S"], w["Dh"], w["seed"])
        return q, k, v, grad_inputs(q.shape, w["seed"])
    if w["kind"] == "chunk":
        q, k, v = prefill_inputs(w["B"], w["Hq"], w["Hkv"], w["Tmax"], w["Dh"], w["seed"])
        return q[:, :, :w["Sq"]].contiguous(), k, v
    return decode_inputs(w["B"], w["Hq"], w["Hkv"], w["Tmax"], w["Dh"], w["lmin"], w["lmax"],
                         w["seed"])
