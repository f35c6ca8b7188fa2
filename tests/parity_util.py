"""Helpers for comparing the CUDA path with the fp64 oracle (test infrastructure)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances the targets state: bf16 inputs with fp32 accumulation, and the fp32 path.
BF16_MAX_ABS = 1e-2
BF16_REL_L2 = 5e-3
F32_MAX_ABS = 1e-4
# fp16 (no stated target; derived from the arithmetic): P and the output are rounded to
# fp16 (11 significant bits, half-ulp 2^-11 relative).  Output rounding is at most
# |o| * 2^-11 <= 5 * 2^-11 ~ 2.4e-3 for N(0, 1) values, and the rounded-P weights move
# an output by at most 2^-11 * max|v - o| ~ 4.4e-3 if every rounding error aligned, so
# max-abs <= 5e-3 covers the sum with margin for fp32 accumulation; the relative L2 of
# random rounding is ~2^-11 / sqrt(3) ~ 3e-4 per term, bounded here by 1e-3.
F16_MAX_ABS = 5e-3
F16_REL_L2 = 1e-3


def errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel_l2 = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel_l2


def assert_close(got, ref, dtype: str, what: str = ""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel_l2 = errors(got, ref)
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {F32_MAX_ABS}"
    elif dtype == "f16":
        assert max_abs <= F16_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {F16_MAX_ABS}"
        assert rel_l2 <= F16_REL_L2, f"{what}: rel-L2 {rel_l2:.3e} > {F16_REL_L2}"
    else:
        assert max_abs <= BF16_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {BF16_MAX_ABS}"
        assert rel_l2 <= BF16_REL_L2, f"{what}: rel-L2 {rel_l2:.3e} > {BF16_REL_L2}"
    return max_abs, rel_l2


def assert_close_per_head(got, ref, dtype: str, what: str = ""):
    """assert_close over the whole output, then the relative-L2 bound again on every (batch,
    head) slab [..., L, D], so that a fault confined to a few CTAs cannot hide in the norm of
    a large tensor (max-abs is already element by element)."""
    res = assert_close(got, ref, dtype, what)
    g = np.asarray(got, dtype=np.float64).reshape(-1, got.shape[-2] * got.shape[-1])
    r = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-2] * ref.shape[-1])
    bound = {"f16": F16_REL_L2, "bf16": BF16_REL_L2}.get(dtype)
    if bound is not None:
        num = np.linalg.norm(g - r, axis=1)
        den = np.linalg.norm(r, axis=1)
        rel = np.where(den > 0, num / np.maximum(den, 1e-300), num)
        worst = int(np.argmax(rel))
        assert rel[worst] <= bound, f"{what}: slab {worst} rel-L2 {rel[worst]:.3e} > {bound}"
    return res


def oracle_rows(q, k, v, rows, *, key_lens=None, **kw):
    """Oracle output for flat rows (b*Hq + h)*Lq + i of a possibly huge problem.

    Rows are grouped by (b, h); each group runs on the sliced single-head
    sub-problem (its query head and its kv head only), which computes the same
    numbers as the full call without converting the whole tensors.
    """
    B, Hq, Lq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), D))
    groups = {}
    for n, r in enumerate(rows):
        bh, i = divmod(int(r), Lq)
        groups.setdefault(bh, []).append((n, i))
    for bh, items in groups.items():
        b, h = divmod(bh, Hq)
        hk = h // G
        kl = None if key_lens is None else key_lens[b:b + 1]
        res = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, hk:hk + 1], v[b:b + 1, hk:hk + 1],
                               key_lens=kl, rows=[i for _, i in items], **kw)
        for (n, _), row in zip(items, res):
            out[n] = row
    return out


def sample_rows(B: int, Hq: int, Lq: int, n: int, seed: int = 0) -> np.ndarray:
    """Rows spread over every (b, h) corner plus random picks, including tile edges."""
    rng = np.random.default_rng(seed)
    picks = set()
    for b in {0, B - 1}:
        for h in {0, Hq - 1}:
            for i in {0, 1, 127, 128, Lq // 2, Lq - 2, Lq - 1}:
                if 0 <= i < Lq:
                    picks.add((b * Hq + h) * Lq + i)
    while len(picks) < n:
        picks.add(int(rng.integers(0, B * Hq * Lq)))
    return np.array(sorted(picks), dtype=np.int64)


def to_numpy_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()
