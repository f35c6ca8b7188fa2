"""GB300-native (sm_103a) multi-head scaled-dot-product attention.

The compute lives in libattn.so (C ABI, include/attn.h): a tcgen05/TMA fused
prefill kernel (head-major, packed and paged layouts), a head_dim-64 prefill on
64-key blocks, a tensor-core decode kernel (contiguous, per-item and paged
caches), a CUDA-core split-KV decode kernel, an fp32 SIMT kernel and the
attention prelude (split QKV, QK norm, RoPE).  This package is the thin Python binding (ctypes; PyTorch supplies device
memory and streams) plus the in-tree build and the seeded synthetic input
generator.
"""
from ._binding import (ATTN_BF16, ATTN_F16, ATTN_ERR_CUDA, ATTN_ERR_INVALID_ARG, ATTN_ERR_TIMEOUT,  # noqa: F401
                       ATTN_ERR_UNSUPPORTED, ATTN_F32, ATTN_OK, EXPORTED, MASK_CAUSAL, MASK_CAUSAL_WINDOW,
                       MASK_NONE, MASK_WINDOW, QK_COPY, QK_NORM_ROPE, QK_ROPE, QK_ROPE_INTERLEAVED, AttnError,
                       attn_decode_caches, attn_decode_caches_noalloc,
                       attn_decode_paged, attn_fwd, attn_fwd_raw, attn_fwd_varlen,
                       attn_fwd_varlen_paged, attn_qkv_prelude, attn_qkv_prelude_caches, check_device_status,
                       last_error, library_path, load, selftest_timeout, sync_status, version)

__all__ = [
    "attn_fwd", "attn_fwd_raw", "attn_fwd_varlen", "attn_fwd_varlen_paged", "attn_decode_caches",
    "attn_decode_caches_noalloc", "attn_decode_paged", "attn_qkv_prelude", "attn_qkv_prelude_caches", "sync_status", "check_device_status",
    "selftest_timeout", "last_error", "version", "load", "library_path", "AttnError",
    "MASK_NONE", "MASK_CAUSAL", "MASK_WINDOW", "MASK_CAUSAL_WINDOW", "ATTN_BF16", "ATTN_F16", "ATTN_F32",
]
