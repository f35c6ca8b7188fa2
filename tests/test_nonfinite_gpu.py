"""Key and value rows that no query of a call can see never reach its output, whatever they
hold: padding past key_lens[b], cache rows past the newest position, rows outside every
query's window band, and unused rows of packed buffers, caches and pages are filled with
NaN, +Inf and -Inf here, and every entry point must still match the fp64 oracle (which
never reads a masked row: a masked key has weight exactly 0, and a row with weight 0 is
skipped in the weighted sum).

Sources of the rule: ripvec-core Driver::build_attn_mask (padded keys are excluded from the
softmax) and realizar cached/attention.rs batched_causal_softmax (hidden positions keep weight
zero).  On the tensor cores a weight of 0 is still multiplied into the value row, and 0 times
Inf or NaN is NaN, so the kernels zero such rows in shared memory before the product.
"""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import MASK_CAUSAL, MASK_CAUSAL_WINDOW, MASK_NONE, MASK_WINDOW
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


def scale_of(D):
    return float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))


def poison_(t, rows):
    """Fill the given rows (indices along dim -2) with NaN, +Inf and -Inf in turn."""
    vals = (float("nan"), float("inf"), float("-inf"))
    for n, r in enumerate(rows):
        t[..., r, :] = vals[n % 3]


def seen_rows(Lq, Lk, P, mode, window, klen):
    """Key rows some query of the call can see (the union of the visible sets)."""
    seen = np.zeros(Lk, dtype=bool)
    for i in range(Lq):
        qp = P + i
        lo, hi = 0, min(klen, Lk)
        if mode == MASK_CAUSAL:
            hi = min(hi, qp + 1)
        elif mode == MASK_WINDOW and window > 0:
            lo, hi = max(lo, qp - window // 2), min(hi, qp + window // 2 + 1)
        elif mode == MASK_CAUSAL_WINDOW:
            hi = min(hi, qp + 1)
            if window > 0:
                lo = max(lo, qp - window + 1)
        if hi > lo:
            seen[lo:hi] = True
    return seen


def fwd_case(B, Hq, Hkv, Lq, Lk, D, P, mode, window, lens, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, Lq, D, generator=g).to(dtype)
    k = torch.randn(B, Hkv, Lk, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, Lk, D, generator=g).to(dtype)
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32)
    poisoned = 0
    for b in range(B):
        klen = Lk if lens is None else max(0, min(Lk, lens[b]))
        unseen = np.nonzero(~seen_rows(Lq, Lk, P, mode, window, klen))[0]
        poison_(k[b], unseen)
        poison_(v[b], unseen)
        poisoned += len(unseen)
    assert poisoned > 0
    return q, k, v, kl


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 2), (128, 4, 2), (128, 3, 1)])
@pytest.mark.parametrize("Lq,Lk,P,mode,window,lens", [
    (300, 300, 0, MASK_NONE, 0, [0, 77, 300, 128, 129]),        # key padding (the encoder workload)
    (200, 700, 100, MASK_CAUSAL, 0, None),                      # cache rows past the newest query
    (250, 700, 0, MASK_CAUSAL, 0, [700, 180, 256, 1, 699]),     # both
    (300, 900, 200, MASK_WINDOW, 128, None),                    # rows before and after every band
    (200, 600, 50, MASK_CAUSAL_WINDOW, 100, [600, 400, 260, 20, 333]),
])
def test_prefill_ignores_unseen_rows(D, Hq, Hkv, Lq, Lk, P, mode, window, lens):
    B = 5 if lens is not None else 2
    q, k, v, kl = fwd_case(B, Hq, Hkv, Lq, Lk, D, P, mode, window, lens, seed=D + Lq + mode)
    sc = scale_of(D)
    out = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), key_lens=None if kl is None else kl.to(DEV),
                        pos_offset=P, mask_mode=mode, window=window, scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = oracle.attention(q, k, v, key_lens=kl, pos_offset=P, mask_mode=mode, window=window, scale=sc)
    assert np.all(np.isfinite(ref))
    assert_close(to_numpy_f64(out), ref, "bf16", f"prefill D={D} G={Hq // Hkv} mode={mode}")


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (16, 2, 128), (8, 4, 64), (4, 4, 128)])
@pytest.mark.parametrize("Lk,P,lens", [
    (5000, 4999, [4999, 1, 2500, 4000]),     # padding past key_lens (tensor-core decode splits the keys)
    (3000, 1700, None),                      # cache rows past the query's position
    (1024, 1023, [1024, 129, 128, 0]),
])
def test_decode_ignores_unseen_rows(Hq, Hkv, D, Lk, P, lens):
    B = 4
    q, k, v, kl = fwd_case(B, Hq, Hkv, 1, Lk, D, P, MASK_CAUSAL, 0, lens, seed=Hq + Lk)
    sc = scale_of(D)
    out = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), key_lens=None if kl is None else kl.to(DEV),
                        pos_offset=P, mask_mode=MASK_CAUSAL, scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = oracle.attention(q, k, v, key_lens=kl, pos_offset=P, mask_mode=MASK_CAUSAL, scale=sc)
    assert_close(to_numpy_f64(out), ref, "bf16", f"decode Hq={Hq} Hkv={Hkv} D={D}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mode", [MASK_NONE, MASK_CAUSAL])
def test_varlen_ignores_rows_after_the_last_sequence(D, mode):
    lens = [300, 129, 1, 200]
    extra = 150
    Hq, Hkv = 4, 2
    g = torch.Generator().manual_seed(D + mode)
    total = sum(lens) + extra
    q = torch.randn(total, Hq, D, generator=g).bfloat16()
    k = torch.randn(total, Hkv, D, generator=g).bfloat16()
    v = torch.randn(total, Hkv, D, generator=g).bfloat16()
    tail = list(range(sum(lens), total))
    poison_(k.transpose(0, 1), tail)
    poison_(v.transpose(0, 1), tail)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    sc = scale_of(D)
    out = torch.zeros_like(q).to(DEV)
    attn.attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), max(lens), out=out, mask_mode=mode, scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    got = to_numpy_f64(out)
    for b in range(len(lens)):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        ref = oracle.attention(q[s0:s1].permute(1, 0, 2)[None], k[s0:s1].permute(1, 0, 2)[None],
                               v[s0:s1].permute(1, 0, 2)[None], mask_mode=mode, scale=sc)
        assert_close(got[s0:s1], ref[0].transpose(1, 0, 2), "bf16", f"varlen seq {b}")


def _decode_items(m, Hq, Hkv, cap, D, lens, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(m, Hq, D, generator=g).bfloat16()
    ks = [torch.randn(Hkv, cap, D, generator=g).bfloat16() for _ in range(m)]
    vs = [torch.randn(Hkv, cap, D, generator=g).bfloat16() for _ in range(m)]
    for i in range(m):
        rows = list(range(max(0, min(cap, lens[i])), cap))
        poison_(ks[i], rows)
        poison_(vs[i], rows)
    return q, ks, vs


def _decode_reference(q, ks, vs, lens, window, scale):
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


@pytest.mark.parametrize("D,G", [(128, 4), (128, 8), (64, 2), (128, 1)])
@pytest.mark.parametrize("window", [0, 200])
def test_decode_caches_ignore_rows_past_kv_lens(D, G, window):
    m, Hkv, cap = 5, 2, 1500
    lens = [1, 37, 700, 1300, 1500]
    q, ks, vs = _decode_items(m, G * Hkv, Hkv, cap, D, lens, seed=D * G + window)
    sc = scale_of(D)
    kl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = attn.attn_decode_caches(q.to(DEV), [k.to(DEV) for k in ks], [v.to(DEV) for v in vs], kl,
                                  sliding_window=window, scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = _decode_reference(q, ks, vs, lens, window, sc)
    assert_close(out.double().cpu().numpy(), ref, "bf16", f"caches D={D} G={G}")


@pytest.mark.parametrize("D,G,page_size", [(128, 4, 16), (128, 8, 64), (64, 2, 7)])
def test_decode_paged_ignores_unused_page_rows(D, G, page_size):
    m, Hkv, cap = 4, 2, 1100
    lens = [1100, 3, 640, 801]
    q, ks, vs = _decode_items(m, G * Hkv, Hkv, cap, D, lens, seed=D + G + page_size)
    max_pages = -(-cap // page_size)
    # scatter the (poisoned-tail) caches into shuffled pages of two pools; unused pages are NaN
    num_pages = m * max_pages + 5
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(7))[: m * max_pages]
    k_pool = torch.full((num_pages, Hkv, page_size, D), float("nan"), dtype=torch.bfloat16)
    v_pool = torch.full_like(k_pool, float("inf"))
    table = perm.view(m, max_pages).to(torch.int32)
    for i in range(m):
        for j in range(max_pages):
            r0, r1 = j * page_size, min(cap, (j + 1) * page_size)
            k_pool[table[i, j], :, : r1 - r0] = ks[i][:, r0:r1]
            v_pool[table[i, j], :, : r1 - r0] = vs[i][:, r0:r1]
    sc = scale_of(D)
    out = attn.attn_decode_paged(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), table.to(DEV),
                                 torch.tensor(lens, dtype=torch.int32, device=DEV), scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    ref = _decode_reference(q, ks, vs, lens, 0, sc)
    assert_close(out.double().cpu().numpy(), ref, "bf16", f"paged D={D} G={G} page={page_size}")
