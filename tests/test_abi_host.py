"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/attn.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from causal_head_self_gb300 import _binding
from causal_head_self_gb300 import build as _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _binding.load()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", src, flags=re.M))
    return names


def test_header_declares_the_bound_symbols():
    assert _declared_symbols() == set(_binding.ABI_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_checked_build_builds_and_exports_every_symbol():
    # the range-checked variant (-DATTN_CHECK) is a separate library with the same ABI
    path = _build.build(check=True)
    assert path.endswith("libattn_sm103a_check.so")
    checked = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(checked, name), name
    checked.attn_error_string.restype = ctypes.c_char_p
    assert checked.attn_error_string(7) == b"ATTN_ERR_CHECK"


def test_error_strings(lib):
    assert _binding.error_string(0) == "ATTN_OK"
    assert _binding.error_string(4) == "ATTN_ERR_TIMEOUT"
    assert _binding.error_string(_binding.ATTN_ERR_CHECK) == "ATTN_ERR_CHECK"
    assert _binding.error_string(99) == "ATTN_ERR_UNKNOWN"
    assert _binding.version() >> 16 == 1


# Argument checks happen before any CUDA call, so fake (aligned, non-null)
# addresses are safe here: nothing is dereferenced or launched.
P = [0x10000, 0x20000, 0x30000, 0x40000]


def fwd(lib, *args, ptrs=P, scale=0.0):
    B, Hq, Hkv, S, Dh, causal, window = args
    return lib.attn_fwd(*ptrs, B, Hq, Hkv, S, Dh, causal, window, scale, None)


@pytest.mark.parametrize("args,code", [
    ((1, 6, 4, 16, 128, 1, 0), _binding.ATTN_ERR_INVALID_ARG),   # Hq % Hkv != 0
    ((1, 4, 0, 16, 128, 1, 0), _binding.ATTN_ERR_INVALID_ARG),   # no K/V head
    ((-1, 4, 4, 16, 128, 1, 0), _binding.ATTN_ERR_INVALID_ARG),  # negative batch
    ((1, 4, 4, 16, 96, 1, 0), _binding.ATTN_ERR_UNSUPPORTED),    # head size
    ((1, 4, 4, 16, 512, 1, 0), _binding.ATTN_ERR_UNSUPPORTED),
    ((1, 4, 4, 16, 128, 0, 8), _binding.ATTN_ERR_INVALID_ARG),   # window without causal
    ((1, 4, 4, 16, 128, 2, 0), _binding.ATTN_ERR_INVALID_ARG),   # causal flag not 0/1
    ((0, 4, 4, 16, 128, 1, 0), _binding.ATTN_OK),                # empty batch: no-op
    ((2, 4, 4, 0, 128, 1, 0), _binding.ATTN_OK),                 # empty sequence: no-op
])
def test_fwd_argument_checks(lib, args, code):
    assert fwd(lib, *args) == code


def test_fwd_rejects_bad_pointers_and_scale(lib):
    a = (1, 4, 4, 16, 128, 1, 0)
    assert fwd(lib, *a, ptrs=[0x10008, *P[1:]]) == _binding.ATTN_ERR_INVALID_ARG   # misaligned
    assert fwd(lib, *a, ptrs=[0, *P[1:]]) == _binding.ATTN_ERR_INVALID_ARG         # null
    assert fwd(lib, *a, ptrs=[P[0], P[1], P[2], P[0]]) == _binding.ATTN_ERR_INVALID_ARG   # o aliases q
    assert fwd(lib, *a, scale=-1.0) == _binding.ATTN_ERR_INVALID_ARG
    assert fwd(lib, *a, scale=float("nan")) == _binding.ATTN_ERR_INVALID_ARG


def test_decode_argument_checks(lib):
    def dec(B, Hq, Hkv, Tmax, Dh, window=0, ptrs=(0x10000, 0x20000, 0x30000, 0x40000, 0x50000),
            scale=0.0):
        return lib.attn_decode(*ptrs, B, Hq, Hkv, Tmax, Dh, window, scale, None)
    assert dec(2, 6, 4, 64, 128) == _binding.ATTN_ERR_INVALID_ARG
    assert dec(2, 8, 4, 0, 128) == _binding.ATTN_ERR_INVALID_ARG
    assert dec(2, 8, 4, 64, 80) == _binding.ATTN_ERR_UNSUPPORTED
    assert dec(0, 8, 4, 64, 128) == _binding.ATTN_OK
    assert dec(2, 8, 4, 64, 128, ptrs=(0x10000, 0x20000, 0x30000, 0x40002, 0x50000)) == \
        _binding.ATTN_ERR_INVALID_ARG   # seqlens not 4-byte aligned
    assert dec(2, 8, 4, 64, 128, scale=-2.0) == _binding.ATTN_ERR_INVALID_ARG


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        _binding.attn_fwd(q, q, q)


def test_fwd_lse_argument_checks(lib):
    a = (1, 4, 4, 16, 128, 1, 0)
    f = lib.attn_fwd_lse
    assert f(*P, None, *a, 0.0, None) == _binding.ATTN_ERR_INVALID_ARG          # no lse
    assert f(*P, 0x50002, *a, 0.0, None) == _binding.ATTN_ERR_INVALID_ARG       # misaligned lse
    assert f(*P, 0x50000, 1, 4, 4, 16, 96, 1, 0, 0.0, None) == _binding.ATTN_ERR_UNSUPPORTED
    assert f(*P, None, 0, 4, 4, 16, 128, 1, 0, 0.0, None) == _binding.ATTN_OK   # empty: no-op
    assert f(*P, 0x10000, *a, 0.0, None) == _binding.ATTN_ERR_INVALID_ARG       # lse aliases q


# q, k, v, o, dout, lse, dq, dk, dv (disjoint fake addresses)
PB = [0x100000 * (i + 1) for i in range(9)]


def bwd(lib, *args, ptrs=PB, scale=0.0):
    B, Hq, Hkv, S, Dh, causal, window = args
    return lib.attn_bwd(*ptrs, B, Hq, Hkv, S, Dh, causal, window, scale, None)


@pytest.mark.parametrize("args,code", [
    ((1, 6, 4, 16, 128, 1, 0), _binding.ATTN_ERR_INVALID_ARG),   # Hq % Hkv != 0
    ((1, 4, 4, 16, 96, 1, 0), _binding.ATTN_ERR_UNSUPPORTED),    # backward takes Dh 64 / 128 / 256
    ((1, 4, 4, 16, 128, 0, 8), _binding.ATTN_ERR_INVALID_ARG),   # window without causal
    ((1, 4, 4, 16, 128, 2, 0), _binding.ATTN_ERR_INVALID_ARG),   # causal flag not 0/1
    ((0, 4, 4, 16, 128, 1, 0), _binding.ATTN_OK),                # empty batch: no-op
    ((2, 4, 4, 0, 128, 1, 0), _binding.ATTN_OK),                 # empty sequence: no-op
])
def test_bwd_argument_checks(lib, args, code):
    assert bwd(lib, *args) == code


def test_bwd_rejects_bad_pointers_aliasing_and_scale(lib):
    a = (1, 4, 4, 16, 128, 1, 0)
    assert bwd(lib, *a, scale=-1.0) == _binding.ATTN_ERR_INVALID_ARG
    assert bwd(lib, *a, ptrs=PB[:5] + [0] + PB[6:]) == _binding.ATTN_ERR_INVALID_ARG        # no lse
    assert bwd(lib, *a, ptrs=PB[:6] + [PB[6] + 8] + PB[7:]) == _binding.ATTN_ERR_INVALID_ARG  # dq misaligned
    assert bwd(lib, *a, ptrs=PB[:6] + [PB[0]] + PB[7:]) == _binding.ATTN_ERR_INVALID_ARG     # dq = q
    assert bwd(lib, *a, ptrs=PB[:7] + [PB[6]] + PB[8:]) == _binding.ATTN_ERR_INVALID_ARG     # dk = dq
