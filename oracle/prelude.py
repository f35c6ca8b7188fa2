"""fp64 reference of the attention prelude: split fused QKV, per-head RMS norm, RoPE,
head-major transpose, optionally straight into a KV cache.

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the bench's CPU baseline may use it;
the product library never calls it and shares no code with it.

What it computes follows ferrum-kernels Backend::split_qkv_norm_rope and
Backend::split_qkv_norm_rope_into_cache, step by step in the order the pages give:

  split      qkv [tokens, q_heads*hd + 2*kv_heads*hd] -> Q, K, V rows of one token
             (Backend::split_qkv: Q first, then K, then V along the feature axis)
  norm       qk_mode 1 only, Q and K: per-head RMS norm over the head's hd values,
             y = x / sqrt(mean(x^2) + eps) * w, one weight vector of hd values per
             projection (q_norm_w, k_norm_w), shared by all heads (Backend::qk_norm_rope,
             mode 1: "per-head RMS norm")
  rope       Q and K, qk_mode 1 and 2: half-split rotation (element j pairs with
             j + hd/2); qk_mode 3: interleaved rotation (element 2j pairs with 2j+1);
             angle index j in [0, hd/2), position pos_offset + t (Backend::qk_norm_rope:
             "positions are taken as pos_offset + i")
  transpose  [tokens, heads, hd] -> [heads, tokens, hd]; V is transpose only
  cache      the _into_cache variant writes K and V at rows [cache_len, cache_len + tokens)
             of [kv_heads, capacity, hd] caches (Backend::kv_cache_append_head_major slot)

Readings where the pages are silent: cos and sin are tables [positions, hd/2] indexed by
the absolute position; the norm weights are hd values per projection; qk_mode 0 is
transpose only (the value qk_norm_rope gives it).  A pair (a, b) rotates to
(a cos - b sin, b cos + a sin).
"""
from __future__ import annotations

import numpy as np

QK_MODE_TRANSPOSE, QK_MODE_NORM_ROPE, QK_MODE_ROPE, QK_MODE_ROPE_INTERLEAVED = 0, 1, 2, 3


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Row-wise RMS norm over the last axis, times w."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_half_split(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """x [..., hd]; cos, sin broadcastable to [..., hd/2]. Pairs (j, j + hd/2)."""
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def rope_interleaved(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """x [..., hd]; pairs (2j, 2j + 1)."""
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = b * cos + a * sin
    return out


def split_qkv_norm_rope(qkv, q_norm_w, k_norm_w, cos, sin, *, q_heads: int, kv_heads: int, head_dim: int,
                        pos_offset: int, eps: float, qk_mode: int):
    """Returns (q [q_heads, tokens, hd], k [kv_heads, tokens, hd], v [kv_heads, tokens, hd]) in fp64."""
    x = _f64(qkv)
    T = x.shape[0]
    hd = head_dim
    if x.shape[1] != (q_heads + 2 * kv_heads) * hd:
        raise ValueError("qkv must be [tokens, (q_heads + 2*kv_heads) * head_dim]")
    q = x[:, :q_heads * hd].reshape(T, q_heads, hd)
    k = x[:, q_heads * hd:(q_heads + kv_heads) * hd].reshape(T, kv_heads, hd)
    v = x[:, (q_heads + kv_heads) * hd:].reshape(T, kv_heads, hd)
    if qk_mode not in (0, 1, 2, 3):
        raise ValueError("qk_mode must be 0, 1, 2 or 3")
    if qk_mode == QK_MODE_NORM_ROPE:
        q = rms_norm(q, _f64(q_norm_w), eps)
        k = rms_norm(k, _f64(k_norm_w), eps)
    if qk_mode in (1, 2, 3):
        c = _f64(cos)[pos_offset:pos_offset + T][:, None, :]  # [T, 1, hd/2]
        s = _f64(sin)[pos_offset:pos_offset + T][:, None, :]
        rot = rope_interleaved if qk_mode == QK_MODE_ROPE_INTERLEAVED else rope_half_split
        q = rot(q, c, s)
        k = rot(k, c, s)
    return q.transpose(1, 0, 2).copy(), k.transpose(1, 0, 2).copy(), v.transpose(1, 0, 2).copy()


def split_qkv_norm_rope_into_cache(qkv, q_norm_w, k_norm_w, cos, sin, cache_k, cache_v, *, q_heads: int,
                                   kv_heads: int, head_dim: int, pos_offset: int, eps: float, qk_mode: int,
                                   cache_len: int):
    """Returns (q [q_heads, tokens, hd], new cache_k, new cache_v) in fp64; the caches are
    [kv_heads, capacity, hd] and only rows [cache_len, cache_len + tokens) change."""
    q, k, v = split_qkv_norm_rope(qkv, q_norm_w, k_norm_w, cos, sin, q_heads=q_heads, kv_heads=kv_heads,
                                  head_dim=head_dim, pos_offset=pos_offset, eps=eps, qk_mode=qk_mode)
    ck, cv = _f64(cache_k).copy(), _f64(cache_v).copy()
    T = q.shape[1]
    if cache_len < 0 or cache_len + T > ck.shape[1]:
        raise ValueError("the new rows must fit the cache capacity")
    ck[:, cache_len:cache_len + T] = k
    cv[:, cache_len:cache_len + T] = v
    return q, ck, cv
