"""GPU parity of the fp16 element type (ATTN_F16) against the fp64 oracle.

The same kernels serve bf16 and fp16; only the operand format of the tensor-core
instructions, the tensor maps and the rounding of P and of the output differ.  The
oracle reads the fp16-rounded inputs.  Tolerance: max-abs <= 5e-3, relative L2 <= 1e-3
(derived from fp16 rounding in tests/parity_util.py).
"""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import (MASK_CAUSAL, MASK_CAUSAL_WINDOW, MASK_NONE, MASK_WINDOW, Case,
                                              WORKLOADS, make_inputs)
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


def check(c: Case, **over):
    q, k, v, kl = make_inputs(c)
    assert q.dtype == torch.float16
    kw = dict(pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window, scale=scale_of(c.D))
    kw.update(over)
    out = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), key_lens=None if kl is None else kl.to(DEV), **kw)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert out.dtype == torch.float16
    ref = oracle.attention(q, k, v, key_lens=kl, **kw)
    return assert_close(to_numpy_f64(out), ref, "f16", c.name)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode,window", [(MASK_NONE, 0), (MASK_CAUSAL, 0), (MASK_WINDOW, 100),
                                         (MASK_CAUSAL_WINDOW, 150)])
@pytest.mark.parametrize("shape", [
    dict(B=2, Hq=4, Hkv=2, Lq=200, Lk=300, pos_offset=100),
    dict(B=2, Hq=3, Hkv=3, Lq=77, Lk=400, pos_offset=0, key_len_range=(0, 400)),
])
def test_prefill_f16(D, mode, window, shape):
    c = Case("f16-prefill", "f16", D=D, mask_mode=mode, window=window, seed=7000 + D + 10 * mode, **shape)
    check(c)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_f16(D, G):
    c = Case("f16-decode", "f16", B=3, Hq=2 * G, Hkv=2, Lq=1, Lk=1000, D=D, pos_offset=999,
             mask_mode=MASK_CAUSAL, seed=7100 + D + G)
    check(c)


def test_prefill_f16_rescaling_and_padding():
    c = Case("f16-big", "f16", B=2, Hq=2, Hkv=1, Lq=256, Lk=640, D=128, mask_mode=MASK_NONE,
             key_len_range=(1, 640), seed=7200)
    check(c, scale=0.6)


def test_causal_gqa_full_size_f16():
    """The causal GQA workload in fp16, every output element against the oracle."""
    base = WORKLOADS["causal_gqa_bf16_4x32q8kv_4096x128"]
    c = Case("causal_gqa_f16_4x32q8kv_4096x128", "f16", B=base.B, Hq=base.Hq, Hkv=base.Hkv, Lq=base.Lq,
             Lk=base.Lk, D=base.D, mask_mode=base.mask_mode, seed=base.seed)
    q, k, v, _ = make_inputs(c)
    out = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), mask_mode=c.mask_mode, scale=scale_of(c.D))
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    got = to_numpy_f64(out)
    del out
    torch.cuda.empty_cache()
    ref = oracle.attention(q, k, v, mask_mode=c.mask_mode, scale=scale_of(c.D))
    assert_close_per_head(got, ref, "f16", c.name)


@pytest.mark.parametrize("window", [0, 300])
def test_decode_caches_f16(window):
    m, Hq, Hkv, cap, D = 4, 8, 2, 900, 128
    lens = [1, 300, 899, 900]
    g = torch.Generator().manual_seed(7300 + window)
    q = torch.randn(m, Hq, D, generator=g).half()
    ks = [torch.randn(Hkv, cap, D, generator=g).half() for _ in range(m)]
    vs = [torch.randn(Hkv, cap, D, generator=g).half() for _ in range(m)]
    kl = torch.tensor(lens, dtype=torch.int32)
    scale = scale_of(D)
    out = attn.attn_decode_caches(q.to(DEV), [t.to(DEV) for t in ks], [t.to(DEV) for t in vs], kl.to(DEV),
                                  sliding_window=window, scale=scale)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert out.dtype == torch.float16
    mode = MASK_CAUSAL_WINDOW if window > 0 else MASK_CAUSAL
    ref = np.stack([oracle.attention(q[i][None, :, None, :], ks[i][None], vs[i][None], pos_offset=lens[i] - 1,
                                     mask_mode=mode, window=window, key_lens=[lens[i]], scale=scale)[0, :, 0, :]
                    for i in range(m)])
    assert_close(out.double().cpu().numpy(), ref, "f16", f"decode caches f16 w={window}")


def test_f16_and_bf16_agree_on_exactly_representable_inputs():
    """Inputs on a coarse grid are exact in both types; the two paths then differ only by
    the rounding of P and of the output (fp16's being the finer)."""
    g = torch.Generator().manual_seed(7400)
    shape_q, shape_kv = (1, 4, 300, 128), (1, 2, 300, 128)
    q = (torch.randint(-8, 9, shape_q, generator=g) / 8.0)
    k = (torch.randint(-8, 9, shape_kv, generator=g) / 8.0)
    v = (torch.randint(-8, 9, shape_kv, generator=g) / 8.0)
    outs = []
    for dt in (torch.float16, torch.bfloat16):
        o = attn.attn_fwd(q.to(DEV, dt), k.to(DEV, dt), v.to(DEV, dt), mask_mode=MASK_CAUSAL, scale=0.1)
        torch.cuda.synchronize()
        outs.append(o.double().cpu())
    ref = oracle.attention(q, k, v, mask_mode=MASK_CAUSAL, scale=0.1)
    assert_close(outs[0].numpy(), ref, "f16", "grid f16")
    assert_close(outs[1].numpy(), ref, "bf16", "grid bf16")
    assert np.max(np.abs(outs[0].numpy() - ref)) <= np.max(np.abs(outs[1].numpy() - ref)) + 1e-3
