"""GB300-native (sm_103a) scaled dot-product causal multi-head self-attention.

The compute path is the CUDA library ``libattn_sm103a.so`` (C ABI in
``include/attn.h``); this package is its thin Python binding.  ``attn_fwd``
runs the tcgen05/TMA prefill kernel, ``attn_decode`` the split-KV decode kernel
with its in-kernel log-sum-exp combine, ``attn_bwd`` the backward pass (given
``attn_fwd_lse``'s output and log-sum-exps).  There is no CPU or PyTorch fallback: without the
built library every call raises.
"""
from ._binding import (ATTN_ERR_CHECK, ATTN_ERR_CUDA, ATTN_ERR_INVALID_ARG, ATTN_ERR_NO_MEMORY,  # noqa: F401
                       ATTN_ERR_SCRATCH_LIMIT, ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED, ATTN_OK,
                       AttnError, attn_bwd, attn_debug_inject_fault, attn_decode,
                       attn_decode_noalloc, attn_decode_ring, attn_fwd, attn_fwd_chunk,
                       attn_fwd_lse, attn_status, error_string, version)
