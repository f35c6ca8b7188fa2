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


@pytest.mark.parametrize("Hq,cap,m", [(4, 900, 4), (8, 900, 4), (16, 900, 4), (8, 5000, 2), (16, 3000, 1)])
def test_decode_caches_agree_with_contiguous_decode(Hq, cap, m):
    """Per-item caches all at full length against attn_fwd over one contiguous cache: both run
    the same kernel with the same split of the keys (the CUDA-core decode at 1 or 2 query heads
    per kv head, the tensor-core decode at 4 and 8, there through one tensor map per item cache
    instead of one over the whole cache), so they agree bit for bit; everything is also checked
    against the oracle."""
    Hkv, D = 2, 128
    q, ks, vs, _ = _case(m, Hq, Hkv, cap, D, [cap] * m, seed=3 + Hq + cap)
    kl = torch.full((m,), cap, dtype=torch.int32, device=DEV)
    a = attn.attn_decode_caches(q.to(DEV), [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], kl)
    k4 = torch.stack(ks).to(DEV)
    v4 = torch.stack(vs).to(DEV)
    b = attn.attn_fwd(q.to(DEV)[:, :, None, :].contiguous(), k4, v4, pos_offset=cap - 1, mask_mode=MASK_CAUSAL)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.equal(a, b[:, :, 0, :])
    ref = oracle.attention(q[:, :, None, :], torch.stack(ks), torch.stack(vs), pos_offset=cap - 1,
                           mask_mode=MASK_CAUSAL, scale=float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32)))
    assert_close(a.double().cpu().numpy(), ref[:, :, 0, :], "bf16", "caches")


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


@pytest.mark.parametrize("cap,offset,m", [(900, 16, 3), (3000, 48, 2), (100, 0, 3), (1000, 0, 3), (5000, 0, 1)])
@pytest.mark.parametrize("window", [0, 333])
@pytest.mark.parametrize("G", [4, 8])
def test_tensor_core_caches_tma(cap, offset, m, window, G):
    """Per-item caches at 4 and 8 query heads per kv head run the tensor-core decode, which
    copies each item's rows by TMA through a K and a V tensor map written on the device for that
    item's address, whatever the caches' alignment beyond 16 bytes, their capacity or the
    lengths.  Without a window the result equals attn_fwd over one contiguous cache with the same
    lengths (the same kernel and split of the keys) bit for bit; every case is also checked
    against the oracle."""
    Hq, Hkv, D = 2 * G, 2, 128
    g = torch.Generator().manual_seed(cap + offset + window + G)
    q = torch.randn(m, Hq, D, generator=g).bfloat16()
    k4 = torch.randn(m, Hkv, cap, D, generator=g).bfloat16()
    v4 = torch.randn(m, Hkv, cap, D, generator=g).bfloat16()
    lens = [cap, max(1, cap // 3), max(1, cap - 7)][:m]
    kd, vd, keep = [], [], []  # each item's cache `offset` bytes into its own allocation
    for i in range(m):
        for src, dst in ((k4[i], kd), (v4[i], vd)):
            buf = torch.empty(src.numel() * 2 + 1024, dtype=torch.uint8, device=DEV)
            view = buf[offset:offset + src.numel() * 2].view(torch.bfloat16).view(Hkv, cap, D)
            view.copy_(src.to(DEV))
            dst.append(view)
            keep.append(buf)
    kl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    sc = float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))
    a = attn.attn_decode_caches(q.to(DEV), kd, vd, kl, sliding_window=window, scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = _reference(q, list(k4), list(v4), kl.cpu(), window, sc)
    assert_close(a.double().cpu().numpy(), ref, "bf16", f"caches cap={cap} offset={offset} w={window}")
    if window == 0:
        # item i's query at position lens[i] - 1 sees positions 0 .. lens[i] - 1: the contiguous
        # decode at pos_offset cap - 1 with key_lens = lens sees the same
        b = attn.attn_fwd(q.to(DEV)[:, :, None, :].contiguous(), k4.to(DEV), v4.to(DEV), key_lens=kl,
                          pos_offset=cap - 1, mask_mode=MASK_CAUSAL, scale=sc)
        torch.cuda.synchronize()
        assert torch.equal(a, b[:, :, 0, :])


@pytest.mark.parametrize("G", [4, 8])
def test_tensor_core_caches_many_items(G):
    """Several hundred items, each with its own K and V maps, ragged lengths including 0 and
    1, fp16, checked against the oracle row by row."""
    m, Hkv, D, cap = 300, 1, 128, 260
    Hq = G * Hkv
    g = torch.Generator().manual_seed(40 + G)
    q = torch.randn(m, Hq, D, generator=g).half()
    ks = [torch.randn(Hkv, cap, D, generator=g).half() for _ in range(m)]
    vs = [torch.randn(Hkv, cap, D, generator=g).half() for _ in range(m)]
    lens = torch.randint(0, cap + 1, (m,), generator=g, dtype=torch.int64).to(torch.int32)
    lens[0], lens[1] = 0, 1
    sc = float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))
    out = attn.attn_decode_caches(q.to(DEV), [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], lens.to(DEV),
                                  scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert out.dtype == torch.float16
    ref = _reference(q, ks, vs, lens, 0, sc)
    assert_close(out.double().cpu().numpy(), ref, "f16", f"many items G={G}")
