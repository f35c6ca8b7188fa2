"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerances: bf16 inputs with fp32 accumulation max-abs <= 1e-2 and relative
L2 <= 5e-3; the fp32 path max-abs <= 1e-4.  The full-size workloads are checked on
every output element; reduced sizes that span several tiles and a ragged tail are
checked in full as well.
"""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import (MASK_CAUSAL, MASK_CAUSAL_WINDOW, MASK_NONE, MASK_WINDOW, Case,
                                              WORKLOADS, case, make_inputs)
from parity_util import assert_close, assert_close_per_head, to_numpy_f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from head_attention_attn_gb300 import build
    build.build_library()
    attn.load()
    yield
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()


def scale_of(D):
    return float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))


def run(c: Case, q, k, v, key_lens, **over):
    kw = dict(pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window, scale=scale_of(c.D))
    kw.update(over)
    out = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV),
                        key_lens=None if key_lens is None else key_lens.to(DEV), **kw)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    return out


def full_check(c: Case, **over):
    q, k, v, kl = make_inputs(c)
    kw = dict(pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window, scale=scale_of(c.D))
    kw.update(over)
    out = run(c, q, k, v, kl, **over)
    ref = oracle.attention(q, k, v, key_lens=kl, **kw)
    return assert_close(to_numpy_f64(out), ref, c.dtype, c.name)


# ------------------------------------------------------------------------------ the five workloads

def test_workload_causal_mha_f32_full():
    full_check(WORKLOADS["causal_mha_f32_1x4x64x32"])


def test_workload_bidir_keypad_bf16_full():
    full_check(WORKLOADS["bidir_keypad_bf16_8x12x512x64"])


@pytest.mark.parametrize("name,small", [
    ("causal_gqa_bf16_4x32q8kv_4096x128", dict(B=1, Hq=8, Hkv=2, Lq=700, Lk=700)),
    ("window128_bf16_4x12x8192x64", dict(B=1, Hq=3, Hkv=3, Lq=1100, Lk=1100)),
    ("decode_bf16_64x32q8kv_8192x128", dict(B=3, Lk=3000, pos_offset=2999)),
])
def test_workloads_reduced_full(name, small):
    full_check(case(name, **small))


_FULL_CACHE = {}


def _full_inputs(name):
    if name not in _FULL_CACHE:
        _FULL_CACHE.clear()
        _FULL_CACHE[name] = make_inputs(WORKLOADS[name])
    return _FULL_CACHE[name]


@pytest.mark.parametrize("name", [
    "causal_gqa_bf16_4x32q8kv_4096x128",
    "window128_bf16_4x12x8192x64",
    "decode_bf16_64x32q8kv_8192x128",
])
def test_workloads_full_size(name):
    """Every output element of the full-size workload against the oracle (the causal GQA
    workload is ~550 GFLOP of fp64 on the host cores), in the launch configuration the bench
    times, plus the relative-L2 bound on every (batch, head) slab."""
    c = WORKLOADS[name]
    q, k, v, kl = _full_inputs(name)
    out = run(c, q, k, v, kl)
    got = to_numpy_f64(out)
    del out
    torch.cuda.empty_cache()
    ref = oracle.attention(q, k, v, key_lens=kl, pos_offset=c.pos_offset, mask_mode=c.mask_mode,
                           window=c.window, scale=scale_of(c.D))
    assert_close_per_head(got, ref, c.dtype, name)


# ------------------------------------------------------------------------------ prefill sweeps (K1)

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode,window", [(MASK_NONE, 0), (MASK_CAUSAL, 0), (MASK_WINDOW, 100),
                                         (MASK_WINDOW, 7), (MASK_CAUSAL_WINDOW, 150), (MASK_CAUSAL_WINDOW, 1)])
@pytest.mark.parametrize("shape", [
    dict(B=2, Hq=4, Hkv=2, Lq=200, Lk=300, pos_offset=100),
    dict(B=1, Hq=2, Hkv=1, Lq=129, Lk=129, pos_offset=0),
    dict(B=2, Hq=3, Hkv=3, Lq=77, Lk=400, pos_offset=0, key_len_range=(0, 400)),
])
def test_prefill_sweep(D, mode, window, shape):
    c = Case("sweep", "bf16", D=D, mask_mode=mode, window=window, seed=D * 100 + mode * 10 + window % 7,
             **shape)
    full_check(c)


@pytest.mark.parametrize("Hq,Hkv", [(3, 1), (6, 2)])
def test_single_query_with_odd_group_uses_prefill(Hq, Hkv):
    c = Case("g3", "bf16", B=2, Hq=Hq, Hkv=Hkv, Lq=1, Lk=333, D=128, pos_offset=332, mask_mode=MASK_CAUSAL,
             seed=5)
    full_check(c)


def test_prefill_scale_zero_and_negative():
    c = Case("sc", "bf16", B=1, Hq=2, Hkv=1, Lq=150, Lk=260, D=64, mask_mode=MASK_CAUSAL, pos_offset=110, seed=6)
    full_check(c, scale=0.0)
    full_check(c, scale=-0.2)


def test_prefill_large_scores_force_rescaling():
    # scale 2.5 makes the running max jump by far more than 2^8 between tiles
    c = Case("big", "bf16", B=1, Hq=2, Hkv=2, Lq=256, Lk=640, D=128, mask_mode=MASK_NONE, seed=7)
    full_check(c, scale=0.6)


def test_paired_head_prefill_scale_zero_and_negative():
    """Head_dim 128 with an even group and no key padding (the persistent form, one CTA per SM
    over the query blocks): scale 0 and a negative scale (the general softmax build)."""
    c = Case("pair_sc", "bf16", B=2, Hq=4, Hkv=2, Lq=300, Lk=420, D=128, mask_mode=MASK_CAUSAL, pos_offset=120, seed=8)
    full_check(c, scale=0.0)
    full_check(c, scale=-0.2)


@pytest.mark.parametrize("Hq", [8, 6])  # even group: the persistent form; odd group: one CTA per block
def test_sharp_softmax_rescaling_within_rounding_bound(Hq):
    """Scale 0.6 at head_dim 128 (about 7x 1/sqrt(128)) makes the running maximum jump by far
    more than 2^8 between key tiles, so O is rescaled in TMEM, and leaves each row's weight on a
    few keys, where the bf16 rounding of P no longer averages out.  bf16 keeps 8 significant
    bits, so each P is within 2^-8 of its value relative, and the row sum adds the same rounded
    values: O moves by at most 2^-8 max|v - O|; rounding O to bf16 adds 2^-8 |O|: in all at
    most 3 * 2^-8 * max|v|.  Both kernels are held to that bound and to the usual relative L2
    bound."""
    c = Case(f"sharp_{Hq}", "bf16", B=1, Hq=Hq, Hkv=2, Lq=600, Lk=900, D=128,
             mask_mode=MASK_NONE, seed=9)
    q, k, v, kl = make_inputs(c)
    out = run(c, q, k, v, kl, scale=0.6)
    ref = oracle.attention(q, k, v, key_lens=kl, mask_mode=c.mask_mode, scale=0.6)
    got = to_numpy_f64(out)
    assert np.all(np.isfinite(got))
    bound = 3 * 2.0 ** -8 * float(v.float().abs().max())
    max_abs = float(np.max(np.abs(got - ref)))
    rel_l2 = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert max_abs <= bound, f"max-abs {max_abs:.3e} > {bound:.3e}"
    assert rel_l2 <= 5e-3, f"rel-L2 {rel_l2:.3e}"


# ------------------------------------------------------------------------------ decode sweeps (K2)

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("Lk,P,mode,window", [
    (1, 0, MASK_CAUSAL, 0), (7, 6, MASK_CAUSAL, 0), (300, 299, MASK_CAUSAL, 0), (2049, 2048, MASK_CAUSAL, 0),
    (1000, 500, MASK_CAUSAL, 0), (3000, 2999, MASK_CAUSAL_WINDOW, 512), (3000, 1500, MASK_WINDOW, 200),
    (640, 0, MASK_NONE, 0),
])
def test_decode_sweep(D, G, Lk, P, mode, window):
    c = Case("dec", "bf16", B=3, Hq=2 * G, Hkv=2, Lq=1, Lk=Lk, D=D, pos_offset=P, mask_mode=mode, window=window,
             seed=G * 1000 + Lk)
    full_check(c)


def test_decode_key_padding_including_empty_rows():
    c = Case("decpad", "bf16", B=6, Hq=8, Hkv=2, Lq=1, Lk=1500, D=128, pos_offset=1499, mask_mode=MASK_CAUSAL,
             seed=8)
    q, k, v, _ = make_inputs(c)
    kl = torch.tensor([0, 1, 17, 1499, 1500, 3000], dtype=torch.int32)  # 3000 clamps to 1500
    out = run(c, q, k, v, kl)
    ref = oracle.attention(q, k, v, key_lens=kl.clamp(0, 1500), pos_offset=1499, mask_mode=MASK_CAUSAL,
                           scale=scale_of(128))
    got = to_numpy_f64(out)
    assert np.all(got[0] == 0.0)
    assert_close(got, ref, "bf16", "decode padding")


# ------------------------------------------------------------------------------ fp32 path (K3)

@pytest.mark.parametrize("D", [1, 5, 32, 64, 100, 256])
@pytest.mark.parametrize("mode,window", [(MASK_NONE, 0), (MASK_CAUSAL, 0), (MASK_WINDOW, 9),
                                         (MASK_CAUSAL_WINDOW, 20)])
def test_f32_sweep(D, mode, window):
    c = Case("f32", "f32", B=2, Hq=4, Hkv=2, Lq=45, Lk=70, D=D, pos_offset=20, mask_mode=mode, window=window,
             key_len_range=(0, 70), seed=D + mode)
    full_check(c)


# ------------------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("dtype,D,Lq", [("bf16", 64, 100), ("bf16", 128, 1), ("f32", 32, 9)])
def test_zero_kv_len_gives_zeros(dtype, D, Lq):
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.randn(2, 4, Lq, D, device=DEV).to(dt)
    k = torch.empty(2, 2, 0, D, device=DEV, dtype=dt)
    out = torch.full_like(q, 7.0)
    attn.attn_fwd(q, k, k, out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


@pytest.mark.parametrize("dtype,D,Lq", [("bf16", 64, 300), ("bf16", 128, 1), ("f32", 16, 30)])
def test_all_keys_padded_gives_zeros(dtype, D, Lq):
    c = Case("pad0", dtype, B=2, Hq=2, Hkv=1, Lq=Lq, Lk=256, D=D, seed=9)
    q, k, v, _ = make_inputs(c)
    out = run(c, q, k, v, torch.zeros(2, dtype=torch.int32))
    assert torch.all(out == 0)


@pytest.mark.parametrize("dtype,D,Lq,mode", [("bf16", 64, 260, MASK_NONE), ("bf16", 128, 1, MASK_CAUSAL),
                                             ("bf16", 128, 200, MASK_CAUSAL), ("f32", 48, 33, MASK_NONE)])
def test_masked_key_values_do_not_leak(dtype, D, Lq, mode):
    c = Case("leak", dtype, B=2, Hq=4, Hkv=2, Lq=Lq, Lk=400, D=D, pos_offset=399 if Lq == 1 else 0,
             mask_mode=mode, seed=10)
    q, k, v, _ = make_inputs(c)
    kl = torch.tensor([300, 123], dtype=torch.int32)
    base = run(c, q, k, v, kl)
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 300:] = 30.0
    v2[0, :, 300:] = -1000.0
    k2[1, :, 123:] = -30.0
    v2[1, :, 123:] = 555.0
    pert = run(c, q, k2, v2, kl)
    assert torch.equal(base, pert)


def test_outputs_outside_the_buffer_are_untouched():
    c = Case("canary", "bf16", B=2, Hq=4, Hkv=2, Lq=130, Lk=190, D=128, mask_mode=MASK_CAUSAL, pos_offset=60,
             seed=11)
    q, k, v, _ = make_inputs(c)
    n = q.numel()
    pad = 4096
    buf = torch.full((n + 2 * pad,), 13.0, dtype=torch.bfloat16, device=DEV)
    out = buf[pad:pad + n].view(q.shape)
    attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), out, pos_offset=60, mask_mode=MASK_CAUSAL)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 13.0) and torch.all(buf[pad + n:] == 13.0)


def test_repeated_calls_are_bitwise_identical():
    c = case("decode_bf16_64x32q8kv_8192x128", B=4, Lk=5000, pos_offset=4999)
    q, k, v, kl = make_inputs(c)
    a = run(c, q, k, v, kl)
    b = run(c, q, k, v, kl)
    assert torch.equal(a, b)
    c = case("causal_gqa_bf16_4x32q8kv_4096x128", B=1, Lq=300, Lk=300)
    q, k, v, kl = make_inputs(c)
    assert torch.equal(run(c, q, k, v, kl), run(c, q, k, v, kl))


def test_runs_on_a_side_stream():
    c = Case("stream", "bf16", B=1, Hq=4, Hkv=1, Lq=256, Lk=256, D=64, mask_mode=MASK_CAUSAL, seed=12)
    q, k, v, _ = make_inputs(c)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = attn.attn_fwd(qd, kd, vd, mask_mode=MASK_CAUSAL)
    s.synchronize()
    ref = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL)
    assert_close(to_numpy_f64(out), ref, "bf16", "side stream")


def test_bounded_wait_times_out_without_faulting():
    assert attn.sync_status() == attn.ATTN_OK
    assert attn.selftest_timeout(2000) == attn.ATTN_OK
    assert attn.sync_status() == attn.ATTN_ERR_TIMEOUT
    assert "timed out" in attn.last_error()
    assert attn.sync_status() == attn.ATTN_OK  # the word is cleared and the context stays usable
    full_check(Case("after", "bf16", B=1, Hq=2, Hkv=1, Lq=64, Lk=64, D=64, seed=13))


# ------------------------------------------------------------------------------ tensor-core decode (K5)

@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("window", [10, 200, 1500])
def test_decode_tc_short_window_leaves_splits_empty(G, window):
    """One batch entry: the split count follows the cache length (up to 4 here), while a short
    window leaves most splits without keys; their empty partials must not disturb the combine."""
    c = Case("dectc", "bf16", B=1, Hq=2 * G, Hkv=2, Lq=1, Lk=8192, D=128, pos_offset=8191,
             mask_mode=MASK_CAUSAL_WINDOW, window=window, seed=9600 + G + window)
    full_check(c)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_decode_tc_key_padding_multi_split(dtype):
    c = Case("dectcpad", dtype, B=4, Hq=32, Hkv=4, Lq=1, Lk=6000, D=128, pos_offset=5999, mask_mode=MASK_CAUSAL,
             key_len_range=(0, 6000), seed=9700)
    full_check(c)


# Windowed masks with more 128-row tiles than the GPU holds at once (four CTAs on each of its
# 152 SMs), so that tiles run in several waves: every output element is compared, with windows
# narrower and wider than a tile, an offset query block, GQA and fp16.
@pytest.mark.parametrize("mode,window,P,extra,dtype", [
    (MASK_WINDOW, 128, 0, 0, "bf16"),
    (MASK_WINDOW, 1, 0, 0, "bf16"),
    (MASK_WINDOW, 300, 0, 0, "bf16"),
    (MASK_WINDOW, 129, 37, 37, "bf16"),
    (MASK_CAUSAL_WINDOW, 200, 0, 0, "bf16"),
    (MASK_CAUSAL_WINDOW, 64, 100, 100, "bf16"),
    (MASK_WINDOW, 128, 0, 0, "f16"),
])
def test_window_band_walk(mode, window, P, extra, dtype):
    c = Case(f"walk_m{mode}_w{window}", dtype, B=2, Hq=8, Hkv=4, Lq=6000, Lk=6000 + extra, D=64, pos_offset=P,
             mask_mode=mode, window=window, seed=700 + window + mode)
    assert (c.Lq + 127) // 128 * c.B * c.Hq > 4 * 152  # more tiles than four CTAs on every SM
    full_check(c)
