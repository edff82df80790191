"""Float64 CPU oracle for causal multi-head self-attention.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The CUDA product path
(``causal_head_self_gb300``) never imports this package, and this package
never imports it: the two share no code.  The seeded input generator
(``causal_head_self_gb300.inputs``) is the one module both sides are fed from,
and it holds none of the attention arithmetic.

What is computed is the definition of scaled dot-product attention from
"Механизм внимания" (llm-arch-research.openidealab.com/textbook/attention),
section "Scaled dot-product attention", written out in ``attn_oracle.c``
(plain C, IEEE double, OpenMP over (batch, head, row block)).  ``brute.py``
holds a second, independent pure-Python restatement for tiny inputs.

Inputs may be torch tensors of any float dtype (bf16 converts to float64
exactly) or numpy arrays; outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (gcc, -fopenmp
    when the compiler has it).  Returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, ip = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, i64,
                                             ip, ip, ip, i64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, dp, dp, dp]
            lib.oracle_attention_bwd.restype = ctypes.c_int
            lib.oracle_attention_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, i64,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_double, ip, i64, ip, i64, dp, dp, dp]
            lib.oracle_softmax_jacobian.restype = ctypes.c_int
            lib.oracle_softmax_jacobian.argtypes = [dp, i64, dp]
            lib.oracle_logsumexp.restype = ctypes.c_double
            lib.oracle_logsumexp.argtypes = [dp, i64]
            lib.oracle_softmax.restype = ctypes.c_int
            lib.oracle_softmax.argtypes = [dp, i64, dp]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().oracle_num_threads())


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def softmax(x) -> np.ndarray:
    """Stable softmax of one row; -inf entries get exactly 0."""
    x = _f64(x).ravel()
    p = np.empty_like(x)
    _load().oracle_softmax(_dp(x), x.size, _dp(p))
    return p


def softmax_jacobian(x) -> np.ndarray:
    """J[i, j] = dp_i / dx_j = p_i (delta_ij - p_j) for p = softmax(x), the
    derivative of section "Почему делить на корень из d_h" of the textbook page."""
    x = _f64(x).ravel()
    J = np.empty((x.size, x.size), np.float64)
    _load().oracle_softmax_jacobian(_dp(x), x.size, _dp(J))
    return J


def logsumexp(x) -> float:
    """log sum_j exp(x_j) of one row (-inf entries contribute 0)."""
    x = _f64(x).ravel()
    return float(_load().oracle_logsumexp(_dp(x), x.size))


def attention(q, k, v, *, causal: bool = True, window: int = 0, window_p4: bool = False,
              scale: float | None = None, rows=None, key_len=None, q_pos0=None,
              return_probs: bool = False, return_lse: bool = False):
    """softmax(Q K^T * scale + M) V for every (batch, query head).

    q: [B, Hq, Sq, Dh]; k, v: [B, Hkv, Skv, Dh] with Hq % Hkv == 0.
    rows: query rows to evaluate (default: all Sq).
    key_len[b]: keys that exist for sequence b (default Skv).
    q_pos0[b]: absolute position of query row 0 (default 0).
    window > 0: key j visible iff i - j < window (window_p4: iff i - j <= window).
    scale None means 1 / sqrt(Dh).
    Returns o [B, Hq, len(rows), Dh], then P [B, Hq, len(rows), Skv] and the
    rows' log-sum-exp of the scaled, masked scores [B, Hq, len(rows)] if asked.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Sq, Dh = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if Bk != B or Dk != Dh or v.shape != k.shape:
        raise ValueError("q/k/v shapes disagree")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if scale is None:
        scale = 1.0 / math.sqrt(Dh)
    rows_a = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = Sq if rows_a is None else rows_a.size
    kl = np.full(B, Skv, np.int64) if key_len is None else np.ascontiguousarray(np.asarray(key_len, np.int64))
    qp = np.zeros(B, np.int64) if q_pos0 is None else np.ascontiguousarray(np.asarray(q_pos0, np.int64))
    out = np.zeros((B, Hq, nrows, Dh), np.float64)
    probs = np.zeros((B, Hq, nrows, Skv), np.float64) if return_probs else None
    lse = np.zeros((B, Hq, nrows), np.float64) if return_lse else None
    rc = _load().oracle_attention(
        _dp(q), _dp(k), _dp(v), B, Hq, Hkv, Sq, Skv, Dh, _ip(kl), _ip(qp),
        _ip(rows_a) if rows_a is not None else None, nrows, int(causal), int(window),
        int(window_p4), float(scale), _dp(out), _dp(probs) if probs is not None else None,
        _dp(lse) if lse is not None else None)
    if rc == -1:
        raise ValueError("oracle_attention rejected its arguments")
    if rc == -2:
        raise ValueError("a query row has no visible key")
    res = (out,) + ((probs,) if return_probs else ()) + ((lse,) if return_lse else ())
    return res if len(res) > 1 else out


def attention_bwd(q, k, v, dout, *, causal: bool = True, window: int = 0,
                  window_p4: bool = False, scale: float | None = None, rows=None, keys=None):
    """Gradients of o = softmax(Q K^T * scale + M) V for a full sequence
    (query row i at position i, S keys): given dout = dL/do, returns
    (dq, dk, dv) = (dL/dq, dL/dk, dL/dv), the chain rule through the
    definition with the softmax Jacobian p_i (delta_ij - p_j).

    q, dout: [B, Hq, S, Dh]; k, v: [B, Hkv, S, Dh].  dk, dv of a K/V head sum
    over the query heads of its group.  rows: dq rows to return (default all);
    keys: dk/dv rows to return (default all; [] for none, which evaluates only
    the given query rows).  dq [B, Hq, len(rows), Dh]; dk, dv [B, Hkv, len(keys), Dh].
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, S, Dh = q.shape
    if k.shape != (B, k.shape[1], S, Dh) or v.shape != k.shape or dout.shape != q.shape:
        raise ValueError("q/k/v/dout shapes disagree")
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if scale is None:
        scale = 1.0 / math.sqrt(Dh)
    rows_a = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    keys_a = None if keys is None else np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    nrows = S if rows_a is None else rows_a.size
    nkeys = S if keys_a is None else keys_a.size
    dq = np.zeros((B, Hq, nrows, Dh), np.float64)
    dk = np.zeros((B, Hkv, nkeys, Dh), np.float64)
    dv = np.zeros((B, Hkv, nkeys, Dh), np.float64)
    rc = _load().oracle_attention_bwd(
        _dp(q), _dp(k), _dp(v), _dp(dout), B, Hq, Hkv, S, Dh, int(causal), int(window),
        int(window_p4), float(scale), _ip(rows_a) if rows_a is not None and rows_a.size else None,
        nrows, _ip(keys_a) if keys_a is not None and keys_a.size else None, nkeys,
        _dp(dq), _dp(dk), _dp(dv))
    if rc == -1:
        raise ValueError("oracle_attention_bwd rejected its arguments")
    if rc == -2:
        raise ValueError("a query row has no visible key")
    return dq, dk, dv


def decode(q, kcache, vcache, seqlens, *, window: int = 0, scale: float | None = None):
    """One KV-cache decode step: the query of sequence b sits at position
    seqlens[b] - 1 and sees cached keys 0 .. seqlens[b] - 1 (the new token's
    own key included), as in section "Prefill и decode" of the textbook page.
    q: [B, Hq, 1, Dh]; caches: [B, Hkv, Tmax, Dh].  Returns [B, Hq, 1, Dh]."""
    sl = np.asarray(seqlens.cpu() if hasattr(seqlens, "cpu") else seqlens, dtype=np.int64)
    return attention(q, kcache, vcache, causal=True, window=window, scale=scale,
                     key_len=sl, q_pos0=sl - 1)
