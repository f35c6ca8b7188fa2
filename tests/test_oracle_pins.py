"""Pins for the fp64 oracle: checks against things other than the oracle itself.

- hand-derived closed forms (tests/golden/closed_forms.json),
- torch's own scaled_dot_product_attention (CPU, fp64) for the special cases
  that reduce to it (bidirectional, key padding, causal, GQA by repetition),
- a separately written pure-Python brute force on tiny inputs,
- invariants the pages fix (rows sum to 1, masked keys weigh exactly 0,
  constant V, q_len 1 at position 0 returns V[0], a window wider than the
  sequence equals the unwindowed mode),
- the banded formulation of ripvec-core Driver::banded_qk / banded_sv,
  re-indexed to the windowed-softmax band, against the dense windowed mode.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from head_attention_attn_gb300.inputs import (MASK_CAUSAL, MASK_CAUSAL_WINDOW, MASK_NONE,
                                              MASK_WINDOW, Case, make_inputs)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _rand(shape, seed, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)


# ----------------------------------------------------------------------------- closed forms

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("gc", _golden_cases(), ids=lambda c: c["name"])
def test_closed_form(gc):
    q = np.array(gc["q"], dtype=np.float32)
    k = np.array(gc["k"], dtype=np.float32)
    v = np.array(gc["v"], dtype=np.float32)
    out = oracle.attention(q, k, v, pos_offset=gc["pos_offset"], mask_mode=gc["mask_mode"],
                           window=gc["window"], key_lens=gc["key_lens"], scale=gc["scale"])
    exp = np.array(gc["expected"], dtype=np.float64)
    assert out.shape == exp.shape
    assert np.max(np.abs(out - exp)) <= gc["tol"]


# ----------------------------------------------------------------------------- library routine

def _sdpa(q, k, v, mask, scale):
    """torch SDPA in fp64 on CPU; GQA by repeating each kv head over its query group."""
    G = q.shape[1] // k.shape[1]
    kk = k.double().repeat_interleave(G, dim=1)
    vv = v.double().repeat_interleave(G, dim=1)
    return F.scaled_dot_product_attention(q.double(), kk, vv, attn_mask=mask, scale=scale)


@pytest.mark.parametrize("B,Hq,Hkv,L,D,seed", [(2, 4, 4, 37, 16, 1), (3, 6, 2, 64, 64, 2),
                                              (1, 8, 1, 129, 32, 3)])
def test_sdpa_bidirectional_key_padding(B, Hq, Hkv, L, D, seed):
    q, k, v = _rand((B, Hq, L, D), seed), _rand((B, Hkv, L, D), seed + 10), _rand((B, Hkv, L, D), seed + 20)
    lens = torch.randint(1, L + 1, (B,), generator=torch.Generator().manual_seed(seed))
    mask = (torch.arange(L)[None, :] < lens[:, None])[:, None, None, :]  # [B,1,1,L] key mask
    scale = 0.37
    ref = _sdpa(q, k, v, mask, scale).numpy()
    out = oracle.attention(q, k, v, mask_mode=MASK_NONE, key_lens=lens.to(torch.int32), scale=scale)
    assert np.max(np.abs(out - ref)) < 1e-10


@pytest.mark.parametrize("B,Hq,Hkv,L,D,seed", [(1, 2, 2, 50, 8, 4), (2, 8, 2, 96, 128, 5)])
def test_sdpa_causal_square(B, Hq, Hkv, L, D, seed):
    q, k, v = _rand((B, Hq, L, D), seed), _rand((B, Hkv, L, D), seed + 1), _rand((B, Hkv, L, D), seed + 2)
    G = Hq // Hkv
    ref = F.scaled_dot_product_attention(q.double(), k.double().repeat_interleave(G, 1),
                                         v.double().repeat_interleave(G, 1), is_causal=True).numpy()
    out = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL)  # default scale 1/sqrt(D) in fp32
    # SDPA uses the exact 1/sqrt(D); the fp32-rounded scale differs by <= 2^-24 relative.
    assert np.max(np.abs(out - ref)) < 1e-6
    out_exact = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, scale=1.0 / math.sqrt(D))
    assert np.max(np.abs(out_exact - ref)) < 1e-10


@pytest.mark.parametrize("Lq,Lk,P", [(5, 12, 7), (1, 33, 32), (16, 16, 0), (8, 40, 20)])
def test_sdpa_causal_with_pos_offset(Lq, Lk, P):
    q, k, v = _rand((2, 4, Lq, 16), 7), _rand((2, 2, Lk, 16), 8), _rand((2, 2, Lk, 16), 9)
    mask = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=P)   # key j visible iff j <= P + i
    ref = _sdpa(q, k, v, mask, 0.25).numpy()
    out = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, pos_offset=P, scale=0.25)
    assert np.max(np.abs(out - ref)) < 1e-10


def test_sdpa_bf16_inputs_are_read_exactly():
    q, k, v = (_rand((1, 2, 20, 64), s, torch.bfloat16) for s in (11, 12, 13))
    ref = _sdpa(q, k, v, None, 0.125).numpy()
    out = oracle.attention(q, k, v, scale=0.125)
    assert np.max(np.abs(out - ref)) < 1e-10


# ----------------------------------------------------------------------------- brute force

def _brute(q, k, v, P, mode, window, lens, scale):
    """Independent pure-Python statement: exclusion set first, then softmax over it."""
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    out = np.zeros((B, Hq, Lq, D))
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            for i in range(Lq):
                pos = P + i
                keep = []
                for j in range(Lk):
                    if lens is not None and j >= lens[b]:
                        continue
                    if mode == MASK_CAUSAL and j > pos:
                        continue
                    if mode == MASK_WINDOW and window and abs(pos - j) > window // 2:
                        continue
                    if mode == MASK_CAUSAL_WINDOW and (j > pos or (window and j <= pos - window)):
                        continue
                    keep.append(j)
                if not keep:
                    continue
                sc = [scale * sum(float(q[b, h, i, d]) * float(k[b, kvh, j, d]) for d in range(D))
                      for j in keep]
                top = max(sc)
                ex = [math.exp(s - top) for s in sc]
                tot = sum(ex)
                for d in range(D):
                    out[b, h, i, d] = sum(e * float(v[b, kvh, j, d]) for e, j in zip(ex, keep)) / tot
    return out


def test_brute_force_exhaustive_tiny():
    n = 0
    for mode, (Lq, Lk), P, (Hq, Hkv), D, lens_kind, window in itertools.product(
            (MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_CAUSAL_WINDOW),
            ((1, 1), (3, 5), (5, 3), (4, 9)), (0, 3), ((1, 1), (2, 1), (4, 2)), (1, 3),
            ("none", "ragged"), (0, 1, 3, 4)):
        if mode in (MASK_NONE, MASK_CAUSAL) and window:
            continue
        B = 2
        seed = n
        q = _rand((B, Hq, Lq, D), seed).numpy()
        k = _rand((B, Hkv, Lk, D), seed + 1000).numpy()
        v = _rand((B, Hkv, Lk, D), seed + 2000).numpy()
        lens = None if lens_kind == "none" else np.array([Lk, max(0, Lk - 2)], dtype=np.int32)
        scale = 0.7
        ref = _brute(q, k, v, P, mode, window, lens, scale)
        out = oracle.attention(q, k, v, pos_offset=P, mask_mode=mode, window=window,
                               key_lens=lens, scale=scale)
        assert np.max(np.abs(out - ref)) < 1e-12, (mode, Lq, Lk, P, Hq, Hkv, D, lens_kind, window)
        n += 1
    assert n > 300


# ----------------------------------------------------------------------------- invariants

ALL_MODES = [(MASK_NONE, 0), (MASK_CAUSAL, 0), (MASK_WINDOW, 6), (MASK_CAUSAL_WINDOW, 5)]


@pytest.mark.parametrize("mode,window", ALL_MODES)
def test_rows_sum_to_one_and_masked_weights_are_zero(mode, window):
    B, Hq, Hkv, Lq, Lk, D, P = 2, 4, 2, 9, 13, 8, 2
    q, k, v = _rand((B, Hq, Lq, D), 21), _rand((B, Hkv, Lk, D), 22), _rand((B, Hkv, Lk, D), 23)
    lens = np.array([13, 6], dtype=np.int32)
    _, w = oracle.attention(q, k, v, pos_offset=P, mask_mode=mode, window=window, key_lens=lens,
                            return_weights=True)
    # One-hot V with scale 0 reveals the visible set (uniform weight over it).
    eye = np.zeros((B, Hkv, Lk, Lk), dtype=np.float32)
    eye[:, :, np.arange(Lk), np.arange(Lk)] = 1.0
    z = np.zeros((B, Hq, Lq, Lk), dtype=np.float32)
    vis = oracle.attention(z, eye, eye, pos_offset=P, mask_mode=mode, window=window, key_lens=lens,
                           scale=0.0) > 0
    for b in range(B):
        for h in range(Hq):
            for i in range(Lq):
                row, seen = w[b, h, i], vis[b, h, i]
                if seen.any():
                    assert abs(row.sum() - 1.0) < 1e-12
                assert np.all(row[~seen] == 0.0)
                assert np.all(row[seen] > 0.0)


@pytest.mark.parametrize("mode,window", ALL_MODES)
def test_visible_set_matches_page_rules(mode, window):
    """scale 0 + one-hot V: output row i = indicator of visible keys / their count."""
    Lq, Lk, P = 7, 12, 3
    lens = np.array([10], dtype=np.int32)
    q = _rand((1, 1, Lq, Lk), 31)
    eye = np.eye(Lk, dtype=np.float32)[None, None]
    out = oracle.attention(q, eye, eye, pos_offset=P, mask_mode=mode, window=window, key_lens=lens,
                           scale=0.0)[0, 0]
    for i in range(Lq):
        pos = P + i
        if mode == MASK_NONE:
            vis = set(range(Lk))
        elif mode == MASK_CAUSAL:
            vis = set(range(0, pos + 1))
        elif mode == MASK_WINDOW:
            vis = set(range(pos - window // 2, pos + window // 2 + 1))
        else:
            vis = set(range(pos - window + 1, pos + 1))
        vis = {j for j in vis if 0 <= j < 10}
        exp = np.zeros(Lk)
        for j in vis:
            exp[j] = 1.0 / len(vis)
        assert np.max(np.abs(out[i] - exp)) < 1e-15


@pytest.mark.parametrize("mode,window", ALL_MODES)
def test_constant_v_returns_constant(mode, window):
    q, k = _rand((2, 4, 6, 16), 41), _rand((2, 2, 10, 16), 42)
    v = np.full((2, 2, 10, 16), 2.5, dtype=np.float32)
    out = oracle.attention(q, k, v, pos_offset=1, mask_mode=mode, window=window)
    assert np.max(np.abs(out - 2.5)) < 1e-13


def test_first_position_causal_returns_v0_exactly():
    q, k, v = _rand((3, 4, 1, 32), 51), _rand((3, 2, 9, 32), 52), _rand((3, 2, 9, 32), 53)
    out = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, pos_offset=0)
    exp = v.double().repeat_interleave(2, dim=1)[:, :, :1, :].numpy()
    assert np.array_equal(out, exp)


def test_single_visible_key_gets_weight_one():
    q, k, v = _rand((1, 1, 1, 8), 55), _rand((1, 1, 4, 8), 56), _rand((1, 1, 4, 8), 57)
    _, w = oracle.attention(q, k, v, mask_mode=MASK_NONE, key_lens=[1], return_weights=True)
    assert w[0, 0, 0, 0] == 1.0 and np.all(w[0, 0, 0, 1:] == 0.0)


def test_wide_windows_equal_unwindowed_modes():
    q, k, v = _rand((2, 2, 11, 8), 61), _rand((2, 2, 17, 8), 62), _rand((2, 2, 17, 8), 63)
    P = 4
    causal = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, pos_offset=P)
    bidir = oracle.attention(q, k, v, mask_mode=MASK_NONE, pos_offset=P)
    for w in (17 + P + 11, 100):
        assert np.array_equal(oracle.attention(q, k, v, mask_mode=MASK_CAUSAL_WINDOW, window=w,
                                               pos_offset=P), causal)
    for w in (2 * (17 + P + 11), 200):
        assert np.array_equal(oracle.attention(q, k, v, mask_mode=MASK_WINDOW, window=w,
                                               pos_offset=P), bidir)
    # window 0 means "no window" in both windowed modes
    assert np.array_equal(oracle.attention(q, k, v, mask_mode=MASK_CAUSAL_WINDOW, window=0,
                                           pos_offset=P), causal)
    assert np.array_equal(oracle.attention(q, k, v, mask_mode=MASK_WINDOW, window=0,
                                           pos_offset=P), bidir)


@pytest.mark.parametrize("mode,window", ALL_MODES)
def test_masked_keys_do_not_influence_output(mode, window):
    B, Hq, Hkv, Lq, Lk, D, P = 2, 2, 1, 6, 12, 8, 2
    q, k, v = _rand((B, Hq, Lq, D), 71), _rand((B, Hkv, Lk, D), 72), _rand((B, Hkv, Lk, D), 73)
    lens = np.array([9, 5], dtype=np.int32)
    base = oracle.attention(q, k, v, pos_offset=P, mask_mode=mode, window=window, key_lens=lens)
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 9:] = 1e3
    v2[0, :, 9:] = -1e3
    k2[1, :, 5:] = -7.0
    v2[1, :, 5:] = 55.0
    pert = oracle.attention(q, k2, v2, pos_offset=P, mask_mode=mode, window=window, key_lens=lens)
    assert np.array_equal(base, pert)


@pytest.mark.parametrize("mode,window", ALL_MODES)
def test_scale_zero_is_mean_of_visible_values(mode, window):
    q, k, v = _rand((1, 1, 5, 4), 81), _rand((1, 1, 8, 4), 82), _rand((1, 1, 8, 4), 83)
    eye = np.eye(8, dtype=np.float32)[None, None]
    z = np.zeros((1, 1, 5, 8), dtype=np.float32)
    weights = oracle.attention(z, eye, eye, pos_offset=2, mask_mode=mode, window=window, scale=0.0)[0, 0]
    out = oracle.attention(q, k, v, pos_offset=2, mask_mode=mode, window=window, scale=0.0)[0, 0]
    assert np.max(np.abs(out - weights @ v[0, 0].double().numpy())) < 1e-13


def test_gqa_equals_mha_with_repeated_kv():
    q, k, v = _rand((2, 8, 7, 16), 91), _rand((2, 2, 11, 16), 92), _rand((2, 2, 11, 16), 93)
    a = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, pos_offset=4)
    b = oracle.attention(q, k.repeat_interleave(4, 1), v.repeat_interleave(4, 1),
                         mask_mode=MASK_CAUSAL, pos_offset=4)
    assert np.array_equal(a, b)


def test_full_key_lens_equals_no_padding():
    q, k, v = _rand((3, 2, 5, 8), 101), _rand((3, 2, 9, 8), 102), _rand((3, 2, 9, 8), 103)
    a = oracle.attention(q, k, v, key_lens=[9, 9, 9])
    b = oracle.attention(q, k, v)
    assert np.array_equal(a, b)


def test_fully_masked_rows_are_zero_not_nan():
    q, k, v = _rand((2, 2, 4, 8), 111), _rand((2, 2, 6, 8), 112), _rand((2, 2, 6, 8), 113)
    out = oracle.attention(q, k, v, key_lens=[0, 6], mask_mode=MASK_CAUSAL)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out))


def test_chunked_prefill_matches_full_prefill():
    q, k, v = _rand((1, 4, 24, 16), 121), _rand((1, 2, 24, 16), 122), _rand((1, 2, 24, 16), 123)
    full = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL)
    a, b = 10, 17
    part = oracle.attention(q[:, :, a:b], k[:, :, :b], v[:, :, :b], mask_mode=MASK_CAUSAL, pos_offset=a)
    assert np.max(np.abs(part - full[:, :, a:b])) < 1e-14


def test_peaked_row_returns_the_matching_value():
    k, v = _rand((1, 1, 10, 32), 131), _rand((1, 1, 10, 32), 132)
    j = 6
    kj = k[0, 0, j].double()
    q = (40.0 * kj / kj.dot(kj)).float()[None, None, None, :]
    out = oracle.attention(q, k, v, scale=1.0)
    assert np.max(np.abs(out[0, 0, 0] - v[0, 0, j].double().numpy())) < 1e-3


def test_rows_api_equals_full_output():
    c = Case("t", "bf16", B=2, Hq=4, Hkv=2, Lq=33, Lk=40, D=16, pos_offset=7, mask_mode=MASK_CAUSAL,
             key_len_range=(1, 40), seed=5)
    q, k, v, lens = make_inputs(c)
    full = oracle.attention(q, k, v, pos_offset=7, mask_mode=MASK_CAUSAL, key_lens=lens)
    rows = [0, 5, 32, 33, 100, 2 * 4 * 33 - 1]
    part = oracle.attention(q, k, v, pos_offset=7, mask_mode=MASK_CAUSAL, key_lens=lens, rows=rows)
    assert np.array_equal(part, full.reshape(-1, 16)[rows])


def test_banded_formulation_matches_dense_window():
    """ripvec-core Driver::banded_qk/banded_softmax/banded_sv indexes keys i - w/2 + t with
    out-of-range slots at -inf; re-indexed to the windowed-softmax band |i-j| <= w/2
    (t in [0, w], i.e. w+1 slots) it must reproduce the dense windowed result."""
    from scipy.special import softmax
    B, H, L, D, w = 2, 3, 40, 8, 10
    q, k, v = _rand((B, H, L, D), 141), _rand((B, H, L, D), 142), _rand((B, H, L, D), 143)
    scale = 0.3
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    half = w // 2
    slots = np.arange(0, w + 1)
    banded = np.zeros((B, H, L, D))
    for i in range(L):
        idx = i - half + slots
        ok = (idx >= 0) & (idx < L)
        sc = np.full((B, H, w + 1), -np.inf)
        sc[:, :, ok] = np.einsum("bhd,bhtd->bht", qd[:, :, i], kd[:, :, idx[ok]])
        p = softmax(sc * scale, axis=-1)
        banded[:, :, i] = np.einsum("bht,bhtd->bhd", p[:, :, ok], vd[:, :, idx[ok]])
    dense = oracle.attention(q, k, v, mask_mode=MASK_WINDOW, window=w, scale=scale)
    assert np.max(np.abs(dense - banded)) < 1e-12


def test_threads_do_not_change_result():
    c = Case("t", "f32", B=2, Hq=4, Hkv=4, Lq=17, Lk=17, D=8, mask_mode=MASK_CAUSAL, seed=9)
    q, k, v, _ = make_inputs(c)
    a = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, nthreads=1)
    b = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, nthreads=5)
    assert np.array_equal(a, b)


def test_rejects_invalid_arguments():
    q, k, v = _rand((1, 3, 4, 8), 1), _rand((1, 2, 4, 8), 2), _rand((1, 2, 4, 8), 3)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v)  # 3 query heads over 2 kv heads
    q = _rand((1, 2, 4, 8), 1)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, mask_mode=7)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, window=-1)
