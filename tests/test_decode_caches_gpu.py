"""Batched decode over per-item KV caches (attn_decode_caches) against the fp64 oracle.

Item i owns caches [Hkv, capacity, D]; its single query is the newest of kv_lens[i]
positions and sees all of them, or the last `sliding_window`.  The oracle computes the
same row as a causal (or causal-window) query at position kv_lens[i]-1 with key padding
kv_lens[i]."""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import MASK_CAUSAL, MASK_CAUSAL_WINDOW
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(m, Hq, Hkv, cap, D, lens, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(m, Hq, D, generator=g).bfloat16()
    ks = [torch.randn(Hkv, cap, D, generator=g).bfloat16() for _ in range(m)]
    vs = [torch.randn(Hkv, cap, D, generator=g).bfloat16() for _ in range(m)]
    return q, ks, vs, torch.tensor(lens, dtype=torch.int32)


def _reference(q, ks, vs, lens, window, scale):
    rows = []
    for i in range(q.shape[0]):
        n = int(min(max(int(lens[i]), 0), ks[i].shape[1]))
        if n == 0:
            rows.append(np.zeros((q.shape[1], q.shape[2])))
            continue
        mode = MASK_CAUSAL_WINDOW if window > 0 else MASK_CAUSAL
        r = oracle.attention(q[i][None, :, None, :], ks[i][None], vs[i][None], pos_offset=n - 1, mask_mode=mode,
                             window=window, key_lens=[n], scale=scale)
        rows.append(r[0, :, 0, :])
    return np.stack(rows)


@pytest.mark.parametrize("D,G", [(128, 4), (128, 1), (64, 8), (64, 2)])
@pytest.mark.parametrize("window", [0, 300])
def test_decode_caches_match_oracle(D, G, window):
    m, Hkv, cap = 5, 2, 1200
    lens = [1, 37, 700, 1200, 1500]  # 1500 clamps to the capacity
    q, ks, vs, kl = _case(m, G * Hkv, Hkv, cap, D, lens, seed=D + G + window)
    scale = float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))
    out = attn.attn_decode_caches(q.to(DEV), [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], kl.to(DEV),
                                  sliding_window=window, scale=scale)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = _reference(q, ks, vs, kl, window, scale)
    assert_close(out.double().cpu().numpy(), ref, "bf16", f"decode caches D={D} G={G} w={window}")


@pytest.mark.parametrize("Hq", [4, 8])
def test_decode_caches_agree_with_contiguous_decode(Hq):
    """Per-item caches all at full length against attn_fwd over one contiguous cache: with
    group 1 or 2 both run the same CUDA-core kernel and agree bit for bit; with group 4 attn_fwd
    runs the tensor-core decode, so both are checked against the oracle instead."""
    m, Hkv, cap, D = 4, 2, 900, 128
    q, ks, vs, _ = _case(m, Hq, Hkv, cap, D, [cap] * m, seed=3)
    kl = torch.full((m,), cap, dtype=torch.int32, device=DEV)
    a = attn.attn_decode_caches(q.to(DEV), [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], kl)
    k4 = torch.stack(ks).to(DEV)
    v4 = torch.stack(vs).to(DEV)
    b = attn.attn_fwd(q.to(DEV)[:, :, None, :].contiguous(), k4, v4, pos_offset=cap - 1, mask_mode=MASK_CAUSAL)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    if Hq // Hkv <= 2:
        assert torch.equal(a, b[:, :, 0, :])
    else:
        ref = oracle.attention(q[:, :, None, :], torch.stack(ks), torch.stack(vs), pos_offset=cap - 1,
                               mask_mode=MASK_CAUSAL, scale=float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32)))
        assert_close(a.double().cpu().numpy(), ref[:, :, 0, :], "bf16", "caches")
        assert_close(b[:, :, 0, :].double().cpu().numpy(), ref[:, :, 0, :], "bf16", "contiguous")


def test_decode_caches_bad_pointer_is_reported_not_read():
    m, Hq, Hkv, cap, D = 2, 4, 1, 256, 128
    q, ks, vs, kl = _case(m, Hq, Hkv, cap, D, [100, 200], seed=4)
    kd = [k.to(DEV) for k in ks]
    vd = [v.to(DEV) for v in vs]
    kp = torch.tensor([kd[0].data_ptr(), kd[1].data_ptr() + 2], dtype=torch.int64, device=DEV)  # misaligned
    vp = torch.tensor([vd[0].data_ptr(), vd[1].data_ptr()], dtype=torch.int64, device=DEV)
    out = torch.full((m, Hq, D), 3.0, dtype=torch.bfloat16, device=DEV)
    st = attn.load().attn_decode_caches(q.to(DEV).data_ptr(), kp.data_ptr(), vp.data_ptr(), out.data_ptr(), m, Hq,
                                        Hkv, cap, D, kl.to(DEV).data_ptr(), 0, 0.1, attn.ATTN_BF16,
                                        torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    assert attn.sync_status() == attn.ATTN_ERR_INVALID_ARG
    assert "misaligned" in attn.last_error() or "aligned" in attn.last_error()
    assert torch.all(out[1] == 0)
    assert attn.sync_status() == attn.ATTN_OK
