"""ctypes binding of libattn.so (include/attn.h): argument marshalling only.

Every step of attention runs in the library's CUDA kernels.  If the library is
missing the first call raises: there is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from .build import LIB_PATH

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_CAUSAL_WINDOW = 0, 1, 2, 3
QK_COPY, QK_NORM_ROPE, QK_ROPE, QK_ROPE_INTERLEAVED = 0, 1, 2, 3
ATTN_BF16, ATTN_F32, ATTN_F16 = 0, 1, 2

EXPORTED = ("attn_fwd", "attn_fwd_out_token_major", "attn_fwd_varlen", "attn_fwd_varlen_paged", "attn_decode_caches",
            "attn_decode_caches_noalloc", "attn_decode_paged", "attn_qkv_prelude", "attn_qkv_prelude_caches", "attn_last_error", "attn_sync_status",
            "attn_selftest_timeout", "attn_version")

_STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
                 4: "ATTN_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A non-OK status from the library; .status holds the attn_status code."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return LIB_PATH


def load(path: str | None = None):
    """Load libattn.so (default: the in-tree build) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libattn.so not found at {p}; build it with "
                               "head_attention_attn_gb300.build.build_library()")
        lib = ctypes.CDLL(p)
        vp, ci = ctypes.c_void_p, ctypes.c_int
        lib.attn_fwd.restype = ci
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, ci, vp, ctypes.c_float, ci, vp]
        lib.attn_fwd_out_token_major.restype = ci
        lib.attn_fwd_out_token_major.argtypes = lib.attn_fwd.argtypes
        lib.attn_fwd_varlen.restype = ci
        lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, ctypes.c_float, ci, vp]
        lib.attn_fwd_varlen_paged.restype = ci
        lib.attn_fwd_varlen_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, ci, ci, ci,
                                              ctypes.c_float, ci, vp]
        lib.attn_qkv_prelude.restype = ci
        lib.attn_qkv_prelude.argtypes = [vp, vp, vp, vp, vp, ci, vp, vp, vp, ci, ci, ci, ci, ci, ctypes.c_float, ci,
                                         ci, ci, ci, vp]
        lib.attn_qkv_prelude_caches.restype = ci
        lib.attn_qkv_prelude_caches.argtypes = [vp, vp, vp, vp, vp, ci, vp, vp, vp, vp, ci, ci, ci, ci, ci,
                                                ctypes.c_float, ci, ci, vp]
        lib.attn_decode_caches.restype = ci
        lib.attn_decode_caches.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, vp, ci, ctypes.c_float, ci, vp]
        lib.attn_decode_caches_noalloc.restype = ci
        lib.attn_decode_caches_noalloc.argtypes = lib.attn_decode_caches.argtypes
        lib.attn_decode_paged.restype = ci
        lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, vp, ci, ctypes.c_float,
                                          ci, vp]
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_last_error.argtypes = []
        lib.attn_sync_status.restype = ci
        lib.attn_sync_status.argtypes = [vp]
        lib.attn_selftest_timeout.restype = ci
        lib.attn_selftest_timeout.argtypes = [ci, vp]
        lib.attn_version.restype = ci
        lib.attn_version.argtypes = []
        if path is None:
            _lib = lib
        return lib


def last_error() -> str:
    return load().attn_last_error().decode()


def _check(status: int):
    if status != ATTN_OK:
        raise AttnError(status, last_error())


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def attn_fwd_raw(q_ptr, k_ptr, v_ptr, out_ptr, batch, q_heads, kv_heads, q_len, kv_len, head_dim,
                 pos_offset, mask_mode, window, key_lens_ptr, scale, dtype, stream_handle) -> int:
    """Direct call of the C entry point with integer pointers; returns the status code."""
    return load().attn_fwd(q_ptr, k_ptr, v_ptr, out_ptr, batch, q_heads, kv_heads, q_len, kv_len, head_dim,
                           pos_offset, mask_mode, window, key_lens_ptr, ctypes.c_float(scale), dtype,
                           stream_handle)


def attn_fwd(q, k, v, out=None, *, pos_offset: int = 0, mask_mode: int = MASK_NONE, window: int = 0,
             key_lens=None, scale: float | None = None, stream=None, out_token_major: bool = False):
    """Attention forward on CUDA tensors (head-major, contiguous).

    q [B, Hq, Lq, D], k and v [B, Hkv, Lk, D] (bf16, fp16 or fp32, same dtype),
    key_lens: int32 CUDA tensor [B] or None; out: preallocated [B, Hq, Lq, D] or None.
    out_token_major: out is [B, Lq, Hq, D] instead (attn_fwd_out_token_major).
    scale None means 1/sqrt(D) rounded to fp32.  Enqueues on `stream`
    (default: torch's current stream) and returns out without synchronising.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share a dtype")
    if q.dtype == torch.bfloat16:
        dtype = ATTN_BF16
    elif q.dtype == torch.float16:
        dtype = ATTN_F16
    elif q.dtype == torch.float32:
        dtype = ATTN_F32
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, Hq, Lq, D = q.shape
    Bk, Hkv, Lk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("shape mismatch between q, k and v")
    out_shape = (B, Lq, Hq, D) if out_token_major else (B, Hq, Lq, D)
    if out is None:
        out = torch.empty(out_shape, dtype=q.dtype, device=q.device)
    elif tuple(out.shape) != out_shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError(f"out must be a contiguous CUDA tensor of shape {out_shape} and q's dtype")
    kl_ptr = None
    if key_lens is not None:
        if key_lens.dtype != torch.int32 or not key_lens.is_cuda or key_lens.numel() != B:
            raise ValueError("key_lens must be an int32 CUDA tensor with B entries")
        kl_ptr = key_lens.data_ptr()
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32).item())
    fn = load().attn_fwd_out_token_major if out_token_major else load().attn_fwd
    status = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, Hq, Hkv, Lq, Lk, D, int(pos_offset),
                int(mask_mode), int(window), kl_ptr, ctypes.c_float(float(scale)), dtype, _stream_handle(stream))
    _check(status)
    return out


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, out=None, *, mask_mode: int = MASK_NONE,
                    window: int = 0, scale: float | None = None, stream=None):
    """Attention over packed sequences (see attn_fwd_varlen in attn.h).

    q [total, Hq, D], k and v [total, Hkv, D]: contiguous bf16 or fp16 CUDA tensors,
    token-major; cu_seqlens: int32 CUDA tensor [batch + 1]; max_seqlen: an upper bound
    on every sequence length.  Returns out [total, Hq, D] without synchronising.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous 3-D CUDA tensor [total, heads, D]")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError("q, k, v must share a dtype")
    if q.dtype == torch.bfloat16:
        dtype = ATTN_BF16
    elif q.dtype == torch.float16:
        dtype = ATTN_F16
    else:
        raise ValueError(f"unsupported dtype {q.dtype} (bf16 or fp16)")
    total, Hq, D = q.shape
    if tuple(k.shape) != tuple(v.shape) or k.shape[0] != total or k.shape[2] != D:
        raise ValueError("k and v must be [total, Hkv, D] matching q")
    Hkv = k.shape[1]
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor [batch + 1]")
    batch = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32).item())
    status = load().attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    cu_seqlens.contiguous().data_ptr(), batch, total, int(max_seqlen), Hq, Hkv, D,
                                    int(mask_mode), int(window), ctypes.c_float(scale), dtype,
                                    _stream_handle(stream))
    _check(status)
    return out


def attn_fwd_varlen_paged(q, k_pool, v_pool, page_table, cu_seqlens, kv_lens, max_seqlen: int, out=None, *,
                          mask_mode: int = MASK_CAUSAL, window: int = 0, scale: float | None = None, stream=None):
    """Packed query chunks against paged caches (see attn_fwd_varlen_paged in attn.h).

    q [total_q, Hq, D] token-major bf16 or fp16; k_pool, v_pool [num_pages, Hkv, page_size, D]
    of q's dtype; page_table int32 [batch, max_pages]; cu_seqlens int32 [batch + 1]; kv_lens
    int32 [batch] (the cached positions, each sequence's queries being the newest of them);
    all contiguous CUDA tensors.  Returns out [total_q, Hq, D] without synchronising.
    """
    import torch
    if not q.is_cuda or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous 3-D CUDA tensor [total_q, q_heads, D]")
    if q.dtype == torch.bfloat16:
        dtype = ATTN_BF16
    elif q.dtype == torch.float16:
        dtype = ATTN_F16
    else:
        raise ValueError(f"unsupported dtype {q.dtype} (bf16 or fp16)")
    total, Hq, D = q.shape
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
        if not t.is_cuda or t.dtype != q.dtype or not t.is_contiguous() or t.dim() != 4 or t.shape[3] != D:
            raise ValueError(f"{name} must be a contiguous CUDA tensor [num_pages, Hkv, page_size, D] of q's dtype")
    if tuple(k_pool.shape) != tuple(v_pool.shape):
        raise ValueError("k_pool and v_pool must share a shape")
    num_pages, Hkv, page_size, _ = (int(x) for x in k_pool.shape)
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1 \
            or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 CUDA tensor [batch + 1]")
    batch = cu_seqlens.numel() - 1
    if page_table.dtype != torch.int32 or not page_table.is_cuda or page_table.dim() != 2 or \
            page_table.shape[0] != batch or not page_table.is_contiguous():
        raise ValueError("page_table must be a contiguous int32 CUDA tensor [batch, max_pages]")
    _check_kv_lens(kv_lens, batch)
    if out is None:
        out = torch.empty_like(q)
    elif tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32).item())
    status = load().attn_fwd_varlen_paged(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), page_table.data_ptr(),
                                          out.data_ptr(), cu_seqlens.data_ptr(), kv_lens.data_ptr(), batch, total,
                                          int(max_seqlen), Hq, Hkv, num_pages, page_size, int(page_table.shape[1]), D,
                                          int(mask_mode), int(window), ctypes.c_float(scale), dtype,
                                          _stream_handle(stream))
    _check(status)
    return out


def attn_qkv_prelude(qkv, q_heads: int, kv_heads: int, head_dim: int, *, qk_mode: int = QK_ROPE, cos=None,
                     sin=None, q_norm_w=None, k_norm_w=None, pos_offset: int = 0, eps: float = 1e-6,
                     q_out=None, k_cache=None, v_cache=None, cache_len: int = 0, stream=None):
    """The attention prelude (see attn_qkv_prelude in attn.h) on CUDA tensors.

    qkv [tokens, (q_heads + 2*kv_heads) * head_dim] bf16 or fp16; cos, sin fp32
    [positions, head_dim/2]; q_norm_w, k_norm_w fp32 [head_dim].  Without caches it
    returns (q [q_heads, tokens, hd], k [kv_heads, tokens, hd], v [kv_heads, tokens, hd]);
    with k_cache/v_cache [kv_heads, capacity, hd] it writes rows cache_len .. cache_len +
    tokens - 1 of them and returns (q, k_cache, v_cache).  Synchronises nothing.
    """
    import torch
    if not qkv.is_cuda or qkv.dim() != 2 or not qkv.is_contiguous():
        raise ValueError("qkv must be a contiguous 2-D CUDA tensor [tokens, features]")
    if qkv.dtype == torch.bfloat16:
        dtype = ATTN_BF16
    elif qkv.dtype == torch.float16:
        dtype = ATTN_F16
    else:
        raise ValueError("qkv must be bf16 or fp16")
    tokens = qkv.shape[0]
    if qkv.shape[1] != (q_heads + 2 * kv_heads) * head_dim:
        raise ValueError("qkv must have (q_heads + 2*kv_heads) * head_dim features")

    def f32(t, name, n=None):
        if t is None:
            return None
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
        if n is not None and t.numel() != n:
            raise ValueError(f"{name} must have {n} values")
        return t

    cos, sin = f32(cos, "cos"), f32(sin, "sin")
    q_norm_w, k_norm_w = f32(q_norm_w, "q_norm_w", head_dim), f32(k_norm_w, "k_norm_w", head_dim)
    positions = 0
    if cos is not None:
        if sin is None or cos.shape != sin.shape or cos.dim() != 2 or cos.shape[1] != head_dim // 2:
            raise ValueError("cos and sin must be [positions, head_dim/2]")
        positions = cos.shape[0]
    if q_out is None:
        q_out = torch.empty((q_heads, tokens, head_dim), dtype=qkv.dtype, device=qkv.device)
    if k_cache is None:
        if v_cache is not None:
            raise ValueError("give both caches or neither")
        k_out = torch.empty((kv_heads, tokens, head_dim), dtype=qkv.dtype, device=qkv.device)
        v_out = torch.empty_like(k_out)
        capacity = 0
    else:
        if v_cache is None or k_cache.shape != v_cache.shape or k_cache.dim() != 3:
            raise ValueError("k_cache and v_cache must be [kv_heads, capacity, head_dim] of one shape")
        if k_cache.shape[0] != kv_heads or k_cache.shape[2] != head_dim or k_cache.dtype != qkv.dtype:
            raise ValueError("caches must be [kv_heads, capacity, head_dim] of qkv's dtype")
        k_out, v_out = k_cache, v_cache
        capacity = k_cache.shape[1]
    ptr = (lambda t: None if t is None else t.data_ptr())
    status = load().attn_qkv_prelude(qkv.data_ptr(), ptr(q_norm_w), ptr(k_norm_w), ptr(cos), ptr(sin), positions,
                                     q_out.data_ptr(), k_out.data_ptr(), v_out.data_ptr(), tokens, q_heads, kv_heads,
                                     head_dim, int(pos_offset), ctypes.c_float(eps), int(qk_mode), int(cache_len),
                                     capacity, dtype, _stream_handle(stream))
    _check(status)
    return q_out, k_out, v_out


def attn_qkv_prelude_caches(qkv, k_caches, v_caches, cache_lens, q_heads: int, kv_heads: int, head_dim: int, *,
                            qk_mode: int = QK_ROPE, cos=None, sin=None, q_norm_w=None, k_norm_w=None,
                            eps: float = 1e-6, q_out=None, capacity: int | None = None, stream=None):
    """Decode-step prelude for m items (see attn_qkv_prelude_caches in attn.h).

    qkv [m, (q_heads + 2*kv_heads) * head_dim] bf16 or fp16; k_caches, v_caches: sequences
    of m [kv_heads, capacity, head_dim] CUDA tensors of qkv's dtype (or int64 CUDA address
    arrays with `capacity` given); cache_lens int32 CUDA [m].  Returns q [m, q_heads, hd].
    """
    import torch
    if not qkv.is_cuda or qkv.dim() != 2 or not qkv.is_contiguous() or qkv.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("qkv must be a contiguous bf16 or fp16 CUDA tensor [m, features]")
    dtype = ATTN_BF16 if qkv.dtype == torch.bfloat16 else ATTN_F16
    m = qkv.shape[0]
    if qkv.shape[1] != (q_heads + 2 * kv_heads) * head_dim:
        raise ValueError("qkv must have (q_heads + 2*kv_heads) * head_dim features")

    def ptrs(caches):
        if isinstance(caches, torch.Tensor) and caches.dtype == torch.int64:
            if capacity is None or caches.numel() != m or not caches.is_cuda:
                raise ValueError("address arrays need m entries on the device and an explicit capacity")
            return caches.contiguous(), int(capacity)
        caches = list(caches)
        if len(caches) != m:
            raise ValueError("one cache per item is required")
        shape = tuple(caches[0].shape)
        for t in caches:
            if (not t.is_cuda or t.dtype != qkv.dtype or not t.is_contiguous() or tuple(t.shape) != shape
                    or len(shape) != 3 or shape[0] != kv_heads or shape[2] != head_dim):
                raise ValueError("caches must be contiguous [kv_heads, capacity, head_dim] tensors of qkv's dtype")
        return torch.tensor([t.data_ptr() for t in caches], dtype=torch.int64, device=qkv.device), shape[1]

    kp, kcap = ptrs(k_caches)
    vp_, vcap = ptrs(v_caches)
    if kcap != vcap:
        raise ValueError("k and v caches must have one capacity")
    if cache_lens.dtype != torch.int32 or not cache_lens.is_cuda or cache_lens.numel() != m:
        raise ValueError("cache_lens must be an int32 CUDA tensor with m entries")
    positions = 0
    if cos is not None:
        if sin is None or cos.shape != sin.shape or cos.dim() != 2 or cos.shape[1] != head_dim // 2:
            raise ValueError("cos and sin must be [positions, head_dim/2]")
        positions = cos.shape[0]
    if q_out is None:
        q_out = torch.empty((m, q_heads, head_dim), dtype=qkv.dtype, device=qkv.device)
    ptr = (lambda t: None if t is None else t.data_ptr())
    status = load().attn_qkv_prelude_caches(qkv.data_ptr(), ptr(q_norm_w), ptr(k_norm_w), ptr(cos), ptr(sin),
                                            positions, q_out.data_ptr(), kp.data_ptr(), vp_.data_ptr(),
                                            cache_lens.data_ptr(), m, q_heads, kv_heads, head_dim, kcap,
                                            ctypes.c_float(eps), int(qk_mode), dtype, _stream_handle(stream))
    _check(status)
    q_out._attn_keepalive = (kp, vp_)
    return q_out


def _check_kv_lens(kv_lens, m: int):
    """kv_lens must be m contiguous int32 values on the device (the kernels index it flat)."""
    import torch
    if not isinstance(kv_lens, torch.Tensor) or kv_lens.dtype != torch.int32 or kv_lens.numel() != m:
        raise ValueError("kv_lens must be an int32 tensor with m entries")
    if not kv_lens.is_contiguous():
        raise ValueError("kv_lens must be contiguous")
    if not kv_lens.is_cuda:
        raise ValueError("kv_lens must be a CUDA tensor")


def _decode_out(q, out):
    """The output of a per-item decode: a new tensor like q, or a checked caller tensor
    (the kernels write m * Hq * D contiguous elements of q's type)."""
    import torch
    if out is None:
        return torch.empty_like(q)
    if not isinstance(out, torch.Tensor) or tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype:
        raise ValueError(f"out must have shape {tuple(q.shape)} and q's dtype {q.dtype}")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    if not out.is_cuda:
        raise ValueError("out must be a CUDA tensor")
    return out


def attn_decode_caches(q, k_caches, v_caches, kv_lens, out=None, *, sliding_window: int = 0,
                       scale: float | None = None, stream=None, kv_heads: int | None = None,
                       capacity: int | None = None, noalloc: bool = False):
    """One decode step for m items against per-item caches (see attn_decode_caches in attn.h;
    noalloc=True calls attn_decode_caches_noalloc instead).

    q: [m, Hq, D] bf16 or fp16 CUDA tensor; k_caches, v_caches: sequences of m
    [Hkv, capacity, D] CUDA tensors of q's dtype, or int64 CUDA tensors of m device
    addresses (then kv_heads and capacity must be given); kv_lens: int32 CUDA [m].
    The pointer arrays are built here (device tensors kept alive until the call is enqueued
    and the stream reaches it; this function synchronises nothing).
    """
    import torch
    if q.dtype == torch.bfloat16:
        dtype = ATTN_BF16
    elif q.dtype == torch.float16:
        dtype = ATTN_F16
    else:
        raise ValueError("q must be bf16 or fp16")
    if not q.is_cuda or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be a contiguous CUDA tensor [m, Hq, D]")
    m, Hq, D = q.shape

    def ptrs(caches):
        if isinstance(caches, torch.Tensor) and caches.dtype == torch.int64:
            if not caches.is_cuda or caches.numel() != m:
                raise ValueError("an address array must be an int64 CUDA tensor with m entries")
            if kv_heads is None or capacity is None:
                raise ValueError("kv_heads and capacity are required with address arrays")
            return caches.contiguous(), (int(kv_heads), int(capacity), D)
        caches = list(caches)
        if len(caches) != m:
            raise ValueError("one cache per item is required")
        shape = tuple(caches[0].shape)
        for t in caches:
            if not t.is_cuda or t.dtype != q.dtype or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError("caches must be contiguous CUDA tensors of q's dtype and one shape [Hkv, capacity, D]")
        arr = torch.tensor([t.data_ptr() for t in caches], dtype=torch.int64, device=q.device)
        return arr, shape

    kp, kshape = ptrs(k_caches)
    vp_, vshape = ptrs(v_caches)
    if len(kshape) != 3 or kshape != vshape or kshape[2] != D:
        raise ValueError("k and v caches must share a shape [Hkv, capacity, D] matching q")
    Hkv, cap = int(kshape[0]), int(kshape[1])
    _check_kv_lens(kv_lens, m)
    out = _decode_out(q, out)
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32).item())
    lib = load()
    entry = lib.attn_decode_caches_noalloc if noalloc else lib.attn_decode_caches
    status = entry(q.data_ptr(), kp.data_ptr(), vp_.data_ptr(), out.data_ptr(), m, Hq, Hkv, cap, D,
                   kv_lens.data_ptr(), int(sliding_window), ctypes.c_float(scale), dtype, _stream_handle(stream))
    _check(status)
    out._attn_keepalive = (kp, vp_)  # the pointer arrays must outlive the queued launch
    return out


def attn_decode_caches_noalloc(q, k_caches, v_caches, kv_lens, out=None, **kw):
    """attn_decode_caches through the entry point that allocates nothing (its tensor maps go to a
    fixed device table of ATTN_NOALLOC_MAX_ITEMS items; calls that overlap on the GPU race)."""
    return attn_decode_caches(q, k_caches, v_caches, kv_lens, out, noalloc=True, **kw)


def attn_decode_paged(q, k_pool, v_pool, page_table, kv_lens, out=None, *, sliding_window: int = 0,
                      scale: float | None = None, stream=None):
    """One decode step for m items over paged caches (see attn_decode_paged in attn.h).

    q: [m, Hq, D] bf16 or fp16 CUDA tensor; k_pool, v_pool: [num_pages, Hkv, page_size, D]
    CUDA tensors of q's dtype; page_table: int32 CUDA [m, max_pages]; kv_lens: int32 CUDA [m].
    Enqueues on `stream` (default: torch's current stream) and returns out.
    """
    import torch
    if q.dtype == torch.bfloat16:
        dtype = ATTN_BF16
    elif q.dtype == torch.float16:
        dtype = ATTN_F16
    else:
        raise ValueError("q must be bf16 or fp16")
    if not q.is_cuda or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be a contiguous CUDA tensor [m, Hq, D]")
    m, Hq, D = q.shape
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
        if not t.is_cuda or t.dtype != q.dtype or not t.is_contiguous() or t.dim() != 4 or t.shape[3] != D:
            raise ValueError(f"{name} must be a contiguous CUDA tensor [num_pages, Hkv, page_size, D] of q's dtype")
    if tuple(k_pool.shape) != tuple(v_pool.shape):
        raise ValueError("k_pool and v_pool must share a shape")
    num_pages, Hkv, page_size, _ = (int(x) for x in k_pool.shape)
    if page_table.dtype != torch.int32 or not page_table.is_cuda or page_table.dim() != 2 or \
            page_table.shape[0] != m or not page_table.is_contiguous():
        raise ValueError("page_table must be a contiguous int32 CUDA tensor [m, max_pages]")
    max_pages = int(page_table.shape[1])
    _check_kv_lens(kv_lens, m)
    out = _decode_out(q, out)
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32).item())
    status = load().attn_decode_paged(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), page_table.data_ptr(),
                                      out.data_ptr(), m, Hq, Hkv, num_pages, page_size, max_pages, D,
                                      kv_lens.data_ptr(), int(sliding_window), ctypes.c_float(scale), dtype,
                                      _stream_handle(stream))
    _check(status)
    return out


def sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device status code."""
    return load().attn_sync_status(_stream_handle(stream))


def check_device_status(stream=None):
    """sync_status(), raising AttnError on a non-OK code."""
    _check(sync_status(stream))


def selftest_timeout(limit_us: int, stream=None) -> int:
    """Enqueue the bounded-wait self test (see attn_selftest_timeout); returns the launch status."""
    return load().attn_selftest_timeout(int(limit_us), _stream_handle(stream))


def version() -> int:
    return load().attn_version()
