"""attn_decode_caches_noalloc: the per-item decode with its tensor maps in the library's fixed
device table instead of a per-call workspace.  Two calls in a row on one stream (the second
rewrites the table the first used) must each equal attn_decode_caches on the same inputs bit
for bit, and the oracle within the bf16 bounds.  This file is collected last."""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import MASK_CAUSAL, MASK_CAUSAL_WINDOW
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MAX_ITEMS = 4096  # ATTN_NOALLOC_MAX_ITEMS


@pytest.fixture(scope="module", autouse=True)
def _library():
    from head_attention_attn_gb300 import build
    build.build_library()
    attn.load()
    yield
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()


def items(m, Hq, Hkv, cap, D, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(m, Hq, D, generator=g).to(dtype)
    ks = [torch.randn(Hkv, cap, D, generator=g).to(dtype) for _ in range(m)]
    vs = [torch.randn(Hkv, cap, D, generator=g).to(dtype) for _ in range(m)]
    lens = torch.randint(0, cap + 1, (m,), generator=g, dtype=torch.int64).to(torch.int32)
    return q, ks, vs, lens


def oracle_rows(q, ks, vs, lens, window, scale):
    rows = []
    for i in range(q.shape[0]):
        n = int(lens[i])
        if n == 0:
            rows.append(np.zeros((q.shape[1], q.shape[2])))
            continue
        mode = MASK_CAUSAL_WINDOW if window > 0 else MASK_CAUSAL
        r = oracle.attention(q[i][None, :, None, :], ks[i][None], vs[i][None], pos_offset=n - 1, mask_mode=mode,
                             window=window, key_lens=[n], scale=scale)
        rows.append(r[0, :, 0, :])
    return np.stack(rows)


@pytest.mark.parametrize("G,D", [(4, 128), (8, 128), (2, 128)])
def test_two_calls_in_a_row_equal_the_allocating_entry(G, D):
    Hkv, cap, window = 2, 700, 0
    sc = float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))
    calls = [items(5, G * Hkv, Hkv, cap, D, seed=70 + G), items(9, G * Hkv, Hkv, cap, D, seed=80 + G)]
    dev = [(q.to(DEV), [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], lens.to(DEV)) for q, ks, vs, lens in calls]
    # both fixed-table calls first, back to back on one stream, then the allocating entry
    fixed = [attn.attn_decode_caches_noalloc(q, ks, vs, lens, sliding_window=window, scale=sc)
             for q, ks, vs, lens in dev]
    ref = [attn.attn_decode_caches(q, ks, vs, lens, sliding_window=window, scale=sc) for q, ks, vs, lens in dev]
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    for i, ((q, ks, vs, lens), a, b) in enumerate(zip(calls, fixed, ref)):
        assert torch.equal(a, b), f"call {i}"
        assert_close(a.double().cpu().numpy(), oracle_rows(q, ks, vs, lens, window, sc), "bf16", f"call {i}")


def test_sliding_window_and_fp16():
    G, Hkv, cap, D, window = 8, 1, 900, 128, 333
    q, ks, vs, lens = items(6, G * Hkv, Hkv, cap, D, seed=90, dtype=torch.float16)
    sc = float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))
    args = (q.to(DEV), [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], lens.to(DEV))
    a = attn.attn_decode_caches_noalloc(*args, sliding_window=window, scale=sc)
    b = attn.attn_decode_caches(*args, sliding_window=window, scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.equal(a, b)
    assert_close(a.double().cpu().numpy(), oracle_rows(q, ks, vs, lens, window, sc), "f16", "window fp16")


def test_the_full_table_and_one_item_more():
    G, Hkv, cap, D = 4, 1, 16, 128
    g = torch.Generator().manual_seed(91)
    m = MAX_ITEMS
    q = torch.randn(m + 1, G * Hkv, D, generator=g).bfloat16().to(DEV)
    k4 = torch.randn(m + 1, Hkv, cap, D, generator=g).bfloat16().to(DEV)
    v4 = torch.randn(m + 1, Hkv, cap, D, generator=g).bfloat16().to(DEV)
    lens = torch.randint(0, cap + 1, (m + 1,), generator=g, dtype=torch.int64).to(torch.int32).to(DEV)
    kp = torch.tensor([k4[i].data_ptr() for i in range(m + 1)], dtype=torch.int64, device=DEV)
    vp = torch.tensor([v4[i].data_ptr() for i in range(m + 1)], dtype=torch.int64, device=DEV)
    kw = dict(scale=0.1, kv_heads=Hkv, capacity=cap)
    a = attn.attn_decode_caches_noalloc(q[:m], kp[:m], vp[:m], lens[:m], **kw)
    b = attn.attn_decode_caches(q[:m], kp[:m], vp[:m], lens[:m], **kw)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.equal(a, b)
    with pytest.raises(attn.AttnError, match="fixed map table"):
        attn.attn_decode_caches_noalloc(q, kp, vp, lens, **kw)
    assert attn.sync_status() == attn.ATTN_OK
