"""GPU parity of attn_fwd_out_token_major: the same attention as attn_fwd with the output
written [B, Lq, Hq, D] (the transposition ferrum-kernels Backend::transpose_head_to_token
applies before the output projection, fused into the store).

Each case checks the token-major output bit for bit against attn_fwd's head-major output
transposed on the host (the same kernels compute both; only the store address differs), and
one case per element type also against the fp64 oracle directly.
"""
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import MASK_CAUSAL, MASK_NONE, MASK_WINDOW, Case, make_inputs
from parity_util import assert_close, to_numpy_f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from head_attention_attn_gb300 import build
    build.build_library()
    attn.load()
    yield
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()


def both(c: Case):
    q, k, v, kl = make_inputs(c)
    kw = dict(pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window,
              key_lens=None if kl is None else kl.to(DEV))
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    head = attn.attn_fwd(qd, kd, vd, **kw)
    tok = attn.attn_fwd(qd, kd, vd, out_token_major=True, **kw)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert tuple(tok.shape) == (c.B, c.Lq, c.Hq, c.D)
    return q, k, v, kl, head, tok


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 128), ("f16", 128), ("f32", 40)])
@pytest.mark.parametrize("shape", [
    dict(B=2, Hq=8, Hkv=2, Lq=300, Lk=300, mask_mode=MASK_CAUSAL),             # even group: paired heads
    dict(B=2, Hq=6, Hkv=2, Lq=200, Lk=330, mask_mode=MASK_WINDOW, window=90),  # odd group: paired row blocks
    dict(B=3, Hq=4, Hkv=4, Lq=130, Lk=257, mask_mode=MASK_NONE, key_len_range=(0, 257)),
    dict(B=2, Hq=8, Hkv=2, Lq=1, Lk=700, pos_offset=699, mask_mode=MASK_CAUSAL),  # decode kernels
])
def test_token_major_equals_transposed_head_major(dtype, D, shape):
    c = Case("tok-out", dtype, D=D, seed=9100 + D + shape["Lq"], **shape)
    _, _, _, _, head, tok = both(c)
    assert torch.equal(tok, head.transpose(1, 2).contiguous())


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64), ("f32", 24)])
def test_token_major_against_oracle(dtype, D):
    c = Case("tok-oracle", dtype, B=2, Hq=4, Hkv=2, Lq=150, Lk=180, D=D, pos_offset=30, mask_mode=MASK_CAUSAL,
             seed=9200 + D)
    q, k, v, kl, _, tok = both(c)
    ref = oracle.attention(q, k, v, key_lens=kl, pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window,
                           scale=float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32)))
    assert_close(to_numpy_f64(tok.transpose(1, 2)), ref, dtype, c.name)


def test_token_major_zero_kv_len_gives_zeros():
    q = torch.randn(2, 4, 5, 64, device=DEV).to(torch.bfloat16)
    k = torch.empty(2, 2, 0, 64, device=DEV, dtype=torch.bfloat16)
    out = torch.full((2, 5, 4, 64), 7.0, device=DEV, dtype=torch.bfloat16)
    attn.attn_fwd(q, k, k, out, out_token_major=True)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
