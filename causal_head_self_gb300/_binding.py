"""ctypes binding of libattn_sm103a.so (include/attn.h), same names as the
C ABI.  Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  torch is used for device memory and streams.

If the library has not been built the first call raises: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# CHS_ATTN_CHECK=1 selects the range-checked build of the same library
# (build.build(check=True)); it runs the same kernels with every copy they
# issue checked, a failed check reported as ATTN_ERR_CHECK
LIB_PATH = os.path.join(_PKG, "libattn_sm103a_check.so" if os.environ.get("CHS_ATTN_CHECK") == "1"
                        else "libattn_sm103a.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_NO_MEMORY = 5
ATTN_ERR_SCRATCH_LIMIT = 6
ATTN_ERR_CHECK = 7

# every symbol include/attn.h declares
ABI_SYMBOLS = ("attn_fwd", "attn_fwd_lse", "attn_fwd_chunk", "attn_bwd", "attn_decode",
               "attn_decode_ring", "attn_decode_noalloc", "attn_status", "attn_error_string",
               "attn_version", "attn_debug_inject_fault")

_lib = None
_lock = threading.Lock()


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} ({code})")


def load():
    """Load (once) and return the ctypes handle of the built library."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.attn_fwd.restype = i
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
            lib.attn_fwd_lse.restype = i
            lib.attn_fwd_lse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
            lib.attn_bwd.restype = i
            lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
            lib.attn_fwd_chunk.restype = i
            lib.attn_fwd_chunk.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp]
            lib.attn_decode.restype = i
            lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
            lib.attn_decode_ring.restype = i
            lib.attn_decode_ring.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
            lib.attn_decode_noalloc.restype = i
            lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
            lib.attn_status.restype = i
            lib.attn_status.argtypes = [vp]
            lib.attn_error_string.restype = ctypes.c_char_p
            lib.attn_error_string.argtypes = [i]
            lib.attn_version.restype = i
            lib.attn_version.argtypes = []
            lib.attn_debug_inject_fault.restype = i
            lib.attn_debug_inject_fault.argtypes = [i]
            _lib = lib
    return _lib


def error_string(code: int) -> str:
    return load().attn_error_string(int(code)).decode()


def version() -> int:
    return int(load().attn_version())


# The current stream's handle without building a torch.cuda.Stream object
# (torch.cuda.current_stream() costs about 3 us per call, a quarter of the
# host's time per library call); the public route where these are missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_current_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream_handle(stream) -> int:
    if stream is None:
        if _raw_stream is not None and _current_device is not None:
            return int(_raw_stream(_current_device()))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_bf16(name, t, ndim):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def attn_fwd(q, k, v, o=None, *, causal=True, window=0, scale=0.0, stream=None):
    """O = softmax(Q K^T * scale + M) V.  q [B,Hq,S,Dh], k/v [B,Hkv,S,Dh] bf16.
    scale 0 means 1/sqrt(Dh).  Returns o (allocated if not given)."""
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, S, Dh = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, S, Dh) or tuple(v.shape) != (B, Hkv, S, Dh):
        raise ValueError("k and v must be [B, Hkv, S, Dh] matching q")
    if o is None:
        o = torch.empty_like(q)
    else:
        _check_bf16("o", o, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    rc = load().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, S,
                         Dh, int(bool(causal)), int(window), float(scale), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return o


def attn_fwd_lse(q, k, v, o=None, lse=None, *, causal=True, window=0, scale=0.0, stream=None):
    """attn_fwd that also returns each row's log-sum-exp lse [B,Hq,S] fp32
    (natural log of the softmax normaliser).  Returns (o, lse)."""
    _check_bf16("q", q, 4)
    _check_bf16("k", k, 4)
    _check_bf16("v", v, 4)
    B, Hq, S, Dh = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, S, Dh) or tuple(v.shape) != (B, Hkv, S, Dh):
        raise ValueError("k and v must be [B, Hkv, S, Dh] matching q")
    if o is None:
        o = torch.empty_like(q)
    else:
        _check_bf16("o", o, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    elif (lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, S) or not lse.is_cuda
          or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous CUDA float32 [B, Hq, S] tensor")
    rc = load().attn_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), B, Hq, Hkv, S, Dh, int(bool(causal)), int(window),
                             float(scale), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_lse")
    return o, lse


def attn_bwd(q, k, v, o, dout, lse, dq=None, dk=None, dv=None, *, causal=True, window=0,
             scale=0.0, stream=None):
    """Backward pass of attn_fwd_lse: (dq, dk, dv) from q, k, v, its output o,
    its lse and dout = dL/do (all as attn_fwd_lse took / returned them)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_bf16(name, t, 4)
    B, Hq, S, Dh = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, S, Dh) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, S, Dh] matching q")
    if o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("o and dout must have q's shape")
    if (lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, S) or not lse.is_cuda
            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous CUDA float32 [B, Hq, S] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _check_bf16(name, t, 4)
        if t.shape != ref.shape:
            raise ValueError(f"{name} must have the shape of its input")
    rc = load().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                         lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv,
                         S, Dh, int(bool(causal)), int(window), float(scale),
                         _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_fwd_chunk(q, kcache, vcache, start_pos, o=None, *, causal=True, window=0, scale=0.0,
                   stream=None):
    """Prefill of one chunk against a KV cache.  q [B,Hq,Sq,Dh]; caches
    [B,Hkv,Tmax,Dh] bf16 already holding the chunk's keys/values at rows
    start_pos .. start_pos+Sq-1.  Query row r sits at position start_pos + r."""
    _check_bf16("q", q, 4)
    _check_bf16("kcache", kcache, 4)
    _check_bf16("vcache", vcache, 4)
    B, Hq, Sq, Dh = q.shape
    Hkv, Tmax = kcache.shape[1], kcache.shape[2]
    if tuple(kcache.shape) != (B, Hkv, Tmax, Dh) or vcache.shape != kcache.shape:
        raise ValueError("the caches must be [B, Hkv, Tmax, Dh] matching q")
    if o is None:
        o = torch.empty_like(q)
    else:
        _check_bf16("o", o, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    rc = load().attn_fwd_chunk(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), o.data_ptr(), B,
                               Hq, Hkv, Sq, Tmax, int(start_pos), Dh, int(bool(causal)),
                               int(window), float(scale), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_chunk")
    return o


def attn_decode(q, kcache, vcache, seqlens, o=None, *, window=0, scale=0.0, stream=None):
    """One decode step.  q [B,Hq,1,Dh]; caches [B,Hkv,Tmax,Dh] bf16; seqlens
    [B] int32 on the device (keys held per sequence, own key included)."""
    _check_bf16("q", q, 4)
    _check_bf16("kcache", kcache, 4)
    _check_bf16("vcache", vcache, 4)
    B, Hq, one, Dh = q.shape
    Hkv, Tmax = kcache.shape[1], kcache.shape[2]
    if one != 1 or tuple(kcache.shape) != (B, Hkv, Tmax, Dh) or vcache.shape != kcache.shape:
        raise ValueError("q must be [B,Hq,1,Dh] and the caches [B,Hkv,Tmax,Dh]")
    if (not isinstance(seqlens, torch.Tensor) or seqlens.dtype != torch.int32 or not seqlens.is_cuda
            or seqlens.numel() != B or not seqlens.is_contiguous()):
        raise TypeError("seqlens must be a contiguous CUDA int32 tensor of B entries")
    if o is None:
        o = torch.empty_like(q)
    else:
        _check_bf16("o", o, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    rc = load().attn_decode(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), seqlens.data_ptr(),
                            o.data_ptr(), B, Hq, Hkv, Tmax, Dh, int(window), float(scale),
                            _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode")
    return o


def attn_decode_ring(q, kcache, vcache, seqlens, o=None, *, window=0, scale=0.0, stream=None):
    """Decode step over a rolling-buffer cache [B,Hkv,C,Dh]: position t of
    sequence b at row t % C; seqlens [B] int32 = tokens so far (see
    include/attn.h)."""
    _check_bf16("q", q, 4)
    _check_bf16("kcache", kcache, 4)
    _check_bf16("vcache", vcache, 4)
    B, Hq, one, Dh = q.shape
    Hkv, C = kcache.shape[1], kcache.shape[2]
    if one != 1 or tuple(kcache.shape) != (B, Hkv, C, Dh) or vcache.shape != kcache.shape:
        raise ValueError("q must be [B,Hq,1,Dh] and the caches [B,Hkv,C,Dh]")
    if (not isinstance(seqlens, torch.Tensor) or seqlens.dtype != torch.int32 or not seqlens.is_cuda
            or seqlens.numel() != B or not seqlens.is_contiguous()):
        raise TypeError("seqlens must be a contiguous CUDA int32 tensor of B entries")
    if o is None:
        o = torch.empty_like(q)
    else:
        _check_bf16("o", o, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    rc = load().attn_decode_ring(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                 seqlens.data_ptr(), o.data_ptr(), B, Hq, Hkv, C, Dh, int(window),
                                 float(scale), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_ring")
    return o


def attn_decode_noalloc(q, kcache, vcache, seqlens, o=None, *, window=0, scale=0.0,
                        stream=None):
    """attn_decode for callers that must not allocate device memory: the
    library's scratch is a fixed 16 MiB device array (see include/attn.h).
    Only the output, when not given, is allocated here by torch."""
    _check_bf16("q", q, 4)
    _check_bf16("kcache", kcache, 4)
    _check_bf16("vcache", vcache, 4)
    B, Hq, one, Dh = q.shape
    Hkv, Tmax = kcache.shape[1], kcache.shape[2]
    if one != 1 or tuple(kcache.shape) != (B, Hkv, Tmax, Dh) or vcache.shape != kcache.shape:
        raise ValueError("q must be [B,Hq,1,Dh] and the caches [B,Hkv,Tmax,Dh]")
    if (not isinstance(seqlens, torch.Tensor) or seqlens.dtype != torch.int32 or not seqlens.is_cuda
            or seqlens.numel() != B or not seqlens.is_contiguous()):
        raise TypeError("seqlens must be a contiguous CUDA int32 tensor of B entries")
    if o is None:
        o = torch.empty_like(q)
    else:
        _check_bf16("o", o, 4)
        if o.shape != q.shape:
            raise ValueError("o must have q's shape")
    rc = load().attn_decode_noalloc(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                    seqlens.data_ptr(), o.data_ptr(), B, Hq, Hkv, Tmax, Dh,
                                    int(window), float(scale), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_noalloc")
    return o


def attn_debug_inject_fault(kind: int) -> None:
    """Test hook (see include/attn.h): 0 none, 1 a prefill K tile is withheld,
    2 a decode key block (CUDA-core path), 3 a decode K tile (tensor-core path);
    later launches wait, give up and report ATTN_ERR_TIMEOUT through attn_status()."""
    rc = load().attn_debug_inject_fault(int(kind))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_debug_inject_fault")


def attn_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device's latched error code."""
    return int(load().attn_status(_stream_handle(stream)))
