"""Packed (unpadded) sequences through attn_fwd_varlen against the fp64 oracle.

Each sequence of the flat token-major batch is its own attention problem; the oracle
computes it on the sequence's rows rearranged to the head-major [1, H, len, D] layout
(the oracle itself is unchanged)."""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import MASK_CAUSAL, MASK_CAUSAL_WINDOW, MASK_NONE, MASK_WINDOW
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from head_attention_attn_gb300 import build
    build.build_library()
    attn.load()
    yield
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()


def packed(lens, Hq, Hkv, D, dtype, seed, extra_rows=0):
    g = torch.Generator().manual_seed(seed)
    total = int(sum(lens)) + extra_rows
    q = torch.randn(total, Hq, D, generator=g).to(dtype)
    k = torch.randn(total, Hkv, D, generator=g).to(dtype)
    v = torch.randn(total, Hkv, D, generator=g).to(dtype)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return q, k, v, cu


def reference(q, k, v, cu, mode, window, scale):
    total, Hq, D = q.shape
    out = np.zeros((total, Hq, D))
    for b in range(cu.numel() - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        qs = q[s0:s1].permute(1, 0, 2)[None]
        ks = k[s0:s1].permute(1, 0, 2)[None]
        vs = v[s0:s1].permute(1, 0, 2)[None]
        r = oracle.attention(qs, ks, vs, mask_mode=mode, window=window, scale=scale)
        out[s0:s1] = r[0].transpose(1, 0, 2)
    return out


def scale_of(D):
    return float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))


LENS = [300, 0, 1, 129, 128, 77, 700, 256]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode,window", [(MASK_NONE, 0), (MASK_CAUSAL, 0), (MASK_WINDOW, 100),
                                         (MASK_CAUSAL_WINDOW, 150)])
def test_varlen_matches_oracle(D, mode, window):
    q, k, v, cu = packed(LENS, 4, 2, D, torch.bfloat16, seed=8000 + D + mode)
    out = attn.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), max(LENS), mask_mode=mode,
                               window=window, scale=scale_of(D))
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = reference(q, k, v, cu, mode, window, scale_of(D))
    assert_close(out.double().cpu().numpy(), ref, "bf16", f"varlen D={D} mode={mode}")


def test_varlen_f16_gqa():
    lens = [500, 3, 260]
    q, k, v, cu = packed(lens, 8, 2, 128, torch.float16, seed=8100)
    out = attn.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), 600, mask_mode=MASK_CAUSAL)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = reference(q, k, v, cu, MASK_CAUSAL, 0, scale_of(128))
    assert_close(out.double().cpu().numpy(), ref, "f16", "varlen f16")


@pytest.mark.parametrize("Hq,Hkv", [(3, 1), (6, 2)])
def test_varlen_odd_group_head_dim_128(Hq, Hkv):
    # an odd group size keeps two consecutive row blocks of one head per CTA (an even one
    # pairs two query heads over the same rows); both layouts are covered for packed rows
    lens = [260, 1, 129, 400]
    q, k, v, cu = packed(lens, Hq, Hkv, 128, torch.bfloat16, seed=8150 + Hq)
    out = attn.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), max(lens), mask_mode=MASK_CAUSAL,
                               scale=scale_of(128))
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = reference(q, k, v, cu, MASK_CAUSAL, 0, scale_of(128))
    assert_close(out.double().cpu().numpy(), ref, "bf16", f"varlen odd group {Hq}/{Hkv}")


def test_varlen_rows_after_the_last_sequence_are_not_written():
    q, k, v, cu = packed([100, 50], 2, 2, 64, torch.bfloat16, seed=8200, extra_rows=30)
    out = torch.full(q.shape, 7.0, dtype=q.dtype, device=DEV)
    attn.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), 100, out=out, mask_mode=MASK_NONE)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.all(out[150:] == 7.0)
    ref = reference(q[:150], k[:150], v[:150], cu, MASK_NONE, 0, scale_of(64))
    assert_close(out[:150].double().cpu().numpy(), ref, "bf16", "varlen head")


def test_varlen_bad_cu_seqlens_is_reported_not_read():
    q, k, v, _ = packed([64, 64], 2, 2, 64, torch.bfloat16, seed=8300)
    cu = torch.tensor([0, 100, 64], dtype=torch.int32, device=DEV)  # decreasing: sequence 1 is invalid
    out = torch.full(q.shape, 5.0, dtype=q.dtype, device=DEV)
    status = attn.load().attn_fwd_varlen(q.to(DEV).data_ptr(), k.to(DEV).data_ptr(), v.to(DEV).data_ptr(),
                                         out.data_ptr(), cu.data_ptr(), 2, 128, 100, 2, 2, 64, MASK_NONE, 0,
                                         0.125, attn.ATTN_BF16, torch.cuda.current_stream().cuda_stream)
    assert status == attn.ATTN_OK
    assert attn.sync_status() == attn.ATTN_ERR_INVALID_ARG
    assert "cu_seqlens" in attn.last_error()
    assert attn.sync_status() == attn.ATTN_OK
    # sequence 0 ([0, 100)) is valid and computed; nothing past row 100 is written
    assert torch.all(out[100:] == 5.0)


@pytest.mark.parametrize("D,mode", [(128, MASK_CAUSAL), (64, MASK_NONE)])
def test_varlen_equal_lengths_equal_attn_fwd(D, mode):
    """All sequences of one length: the packed call and the head-major call compute the
    same numbers (same tiles, same order), only the memory layout differs."""
    B, L, Hq, Hkv = 3, 333, 4, 2
    q, k, v, cu = packed([L] * B, Hq, Hkv, D, torch.bfloat16, seed=8400 + D)
    a = attn.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), L, mask_mode=mode)
    qh = q.view(B, L, Hq, D).permute(0, 2, 1, 3).contiguous().to(DEV)
    kh = k.view(B, L, Hkv, D).permute(0, 2, 1, 3).contiguous().to(DEV)
    vh = v.view(B, L, Hkv, D).permute(0, 2, 1, 3).contiguous().to(DEV)
    b = attn.attn_fwd(qh, kh, vh, mask_mode=mode)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.equal(a.view(B, L, Hq, D).permute(0, 2, 1, 3), b)
