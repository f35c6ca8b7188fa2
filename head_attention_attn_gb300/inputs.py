"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module holds shapes, seeds and random draws only: no attention arithmetic.
It imports neither the oracle nor the CUDA library.

Draw order for every case: Q, K, V as float32 N(0, 1) from one CPU generator,
then a cast to the case's dtype (bf16 or fp16 rounding happens once, and both
the oracle and the kernels read the rounded values), then the per-sequence valid
key lengths when the case has key padding.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Tuple

import torch

MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_CAUSAL_WINDOW = 0, 1, 2, 3


@dataclass(frozen=True)
class Case:
    name: str
    dtype: str            # "bf16", "f16" or "f32"
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    D: int
    pos_offset: int = 0
    mask_mode: int = MASK_NONE
    window: int = 0
    key_len_range: Optional[Tuple[int, int]] = None   # inclusive [lo, hi] for uniform lengths
    seed: int = 0

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[self.dtype]


# The five workloads the pages' encoder, prefill and decode paths are measured on.
WORKLOADS = {
    "causal_mha_f32_1x4x64x32": Case(
        "causal_mha_f32_1x4x64x32", "f32", B=1, Hq=4, Hkv=4, Lq=64, Lk=64, D=32,
        mask_mode=MASK_CAUSAL, seed=1000),
    "bidir_keypad_bf16_8x12x512x64": Case(
        "bidir_keypad_bf16_8x12x512x64", "bf16", B=8, Hq=12, Hkv=12, Lq=512, Lk=512, D=64,
        mask_mode=MASK_NONE, key_len_range=(64, 512), seed=1001),
    "causal_gqa_bf16_4x32q8kv_4096x128": Case(
        "causal_gqa_bf16_4x32q8kv_4096x128", "bf16", B=4, Hq=32, Hkv=8, Lq=4096, Lk=4096, D=128,
        mask_mode=MASK_CAUSAL, seed=1002),
    "window128_bf16_4x12x8192x64": Case(
        "window128_bf16_4x12x8192x64", "bf16", B=4, Hq=12, Hkv=12, Lq=8192, Lk=8192, D=64,
        mask_mode=MASK_WINDOW, window=128, seed=1003),
    "decode_bf16_64x32q8kv_8192x128": Case(
        "decode_bf16_64x32q8kv_8192x128", "bf16", B=64, Hq=32, Hkv=8, Lq=1, Lk=8192, D=128,
        pos_offset=8191, mask_mode=MASK_CAUSAL, seed=1004),
}

WORKLOAD_ORDER = list(WORKLOADS)


def case(name: str, **changes) -> Case:
    """A named workload, optionally with fields replaced (e.g. a smaller size)."""
    return replace(WORKLOADS[name], **changes)


def make_inputs(c: Case, device="cpu"):
    """Seeded q [B,Hq,Lq,D], k, v [B,Hkv,Lk,D] in c's dtype, and key_lens [B] int32 or None."""
    g = torch.Generator("cpu")
    g.manual_seed(int(c.seed))
    dt = c.torch_dtype
    q = torch.randn((c.B, c.Hq, c.Lq, c.D), generator=g, dtype=torch.float32).to(dt)
    k = torch.randn((c.B, c.Hkv, c.Lk, c.D), generator=g, dtype=torch.float32).to(dt)
    v = torch.randn((c.B, c.Hkv, c.Lk, c.D), generator=g, dtype=torch.float32).to(dt)
    key_lens = None
    if c.key_len_range is not None:
        lo, hi = c.key_len_range
        key_lens = torch.randint(lo, hi + 1, (c.B,), generator=g, dtype=torch.int64).to(torch.int32)
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
        if key_lens is not None:
            key_lens = key_lens.to(device)
    return q, k, v, key_lens

