"""Packed multi-token query chunks against paged KV caches (attn_fwd_varlen_paged).

Sequence b has len_b packed queries, the newest of its kv_lens[b] cached positions (chunked
prefill, multi-token verification); its cache lives in pages of two pools addressed by
page_table[b].  Gathering the pages back into one [Hkv, capacity, D] cache and calling attn_fwd
per sequence (q_len len_b, pos_offset kv_lens[b] - len_b, key_lens kv_lens[b]) runs the same
prefill kernel at head_dim 128; where both split the keys into the same 128-key tiles (a causal
mask, whose band starts at key 0, or page sizes gathered row by row) they agree bit for bit.
Page sizes that TMA copies a page at a time start the tiles on multiples of 128, so with a
window the split can differ and the results agree to rounding.  Both are checked against the
fp64 oracle.  Pool rows outside every sequence's cached positions hold NaN, which
must never reach the output.
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


def paged_chunks(q_lens, kv_lens, Hq, Hkv, D, page_size, seed, dtype=torch.bfloat16, spare_pages=5):
    """Packed queries, per-sequence caches scattered over shuffled pool pages (unused rows NaN)."""
    g = torch.Generator().manual_seed(seed)
    B = len(q_lens)
    max_pages = max(1, -(-max(kv_lens) // page_size))
    cap = max_pages * page_size
    total = int(sum(q_lens))
    q = torch.randn(total, Hq, D, generator=g).to(dtype)
    caches_k = torch.randn(B, Hkv, cap, D, generator=g).to(dtype)
    caches_v = torch.randn(B, Hkv, cap, D, generator=g).to(dtype)
    for b in range(B):  # positions past kv_lens[b] hold NaN in the gathered view too
        caches_k[b, :, kv_lens[b]:] = float("nan")
        caches_v[b, :, kv_lens[b]:] = float("nan")
    num_pages = B * max_pages + spare_pages
    perm = torch.randperm(num_pages, generator=g)[: B * max_pages]
    table = perm.view(B, max_pages).to(torch.int32)
    k_pool = torch.full((num_pages, Hkv, page_size, D), float("nan"), dtype=dtype)
    v_pool = torch.full_like(k_pool, float("nan"))
    for b in range(B):
        for j in range(max_pages):
            k_pool[table[b, j]] = caches_k[b, :, j * page_size:(j + 1) * page_size]
            v_pool[table[b, j]] = caches_v[b, :, j * page_size:(j + 1) * page_size]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    return q, k_pool, v_pool, table, cu, torch.tensor(kv_lens, dtype=torch.int32), caches_k, caches_v


def run_paged(q, k_pool, v_pool, table, cu, kl, mode, window, sc, out=None):
    out = attn.attn_fwd_varlen_paged(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), table.to(DEV), cu.to(DEV),
                                     kl.to(DEV), int((cu[1:] - cu[:-1]).max()), out=out, mask_mode=mode,
                                     window=window, scale=sc)
    torch.cuda.synchronize()
    return out


CASES = [
    # q_lens, kv_lens: chunks that straddle pages, a whole prefill, one-token and empty chunks
    ([100, 300, 1, 0, 129, 64], [137, 300, 1000, 50, 700, 64]),
]


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 4, 2), (128, 4, 2), (128, 3, 1), (128, 8, 1)])
# TMA page pieces: 8 (the smallest), 16, 128 (one key tile), 384 (three tiles a page); gathered: 7, 1, 24
@pytest.mark.parametrize("page_size", [8, 16, 128, 384, 7, 1, 24])
@pytest.mark.parametrize("mode,window", [(MASK_CAUSAL, 0), (MASK_CAUSAL_WINDOW, 150)])
def test_paged_chunks_equal_gathered_prefill(D, Hq, Hkv, page_size, mode, window):
    q_lens, kv_lens = CASES[0]
    q, kp, vp, table, cu, kl, ck, cv = paged_chunks(q_lens, kv_lens, Hq, Hkv, D, page_size,
                                                    seed=D + Hq * 10 + page_size + mode)
    sc = scale_of(D)
    out = run_paged(q, kp, vp, table, cu, kl, mode, window, sc)
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    got = to_numpy_f64(out)
    for b, (n, klen) in enumerate(zip(q_lens, kv_lens)):
        if n == 0:
            continue
        s0 = int(cu[b])
        qb = q[s0:s0 + n].permute(1, 0, 2)[None].contiguous()        # [1, Hq, n, D]
        kb, vb = ck[b:b + 1], cv[b:b + 1]                           # [1, Hkv, cap, D]
        P = klen - n
        ref = oracle.attention(qb, kb, vb, pos_offset=P, mask_mode=mode, window=window, key_lens=[klen], scale=sc)
        assert_close(got[s0:s0 + n], ref[0].transpose(1, 0, 2), "bf16", f"seq {b} (len {n}, kv {klen})")
        same_tiles = mode == MASK_CAUSAL or page_size in (7, 1, 24)
        if n > 1 and D == 128 and same_tiles:  # the same prefill kernel and key tiles through attn_fwd: bit for bit
            # (at head_dim 64 attn_fwd runs the 64-key-block kernel, a different summation order)
            fwd = attn.attn_fwd(qb.to(DEV), kb.to(DEV), vb.to(DEV), key_lens=torch.tensor([klen], dtype=torch.int32,
                                device=DEV), pos_offset=P, mask_mode=mode, window=window, scale=sc)
            torch.cuda.synchronize()
            assert torch.equal(fwd[0].transpose(0, 1).cpu(), out[s0:s0 + n].cpu()), f"seq {b}"
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()


@pytest.mark.parametrize("D,page_size", [(128, 32), (64, 64), (128, 13)])
@pytest.mark.parametrize("mode,window", [(MASK_NONE, 0), (MASK_WINDOW, 64)])
def test_paged_chunks_other_masks_against_oracle(mode, window, D, page_size):
    q_lens, kv_lens = [50, 200, 7], [90, 200, 400]
    Hq, Hkv = 4, 2
    q, kp, vp, table, cu, kl, ck, cv = paged_chunks(q_lens, kv_lens, Hq, Hkv, D, page_size, seed=11 + mode + D)
    sc = scale_of(D)
    got = to_numpy_f64(run_paged(q, kp, vp, table, cu, kl, mode, window, sc))
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    for b, (n, klen) in enumerate(zip(q_lens, kv_lens)):
        s0 = int(cu[b])
        ref = oracle.attention(q[s0:s0 + n].permute(1, 0, 2)[None], ck[b:b + 1], cv[b:b + 1], pos_offset=klen - n,
                               mask_mode=mode, window=window, key_lens=[klen], scale=sc)
        assert_close(got[s0:s0 + n], ref[0].transpose(1, 0, 2), "bf16", f"seq {b}")


def test_paged_chunks_f16():
    q_lens, kv_lens = [130, 5], [500, 5]
    q, kp, vp, table, cu, kl, ck, cv = paged_chunks(q_lens, kv_lens, 8, 2, 128, 16, seed=12, dtype=torch.float16)
    sc = scale_of(128)
    out = run_paged(q, kp, vp, table, cu, kl, MASK_CAUSAL, 0, sc)
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert out.dtype == torch.float16
    got = to_numpy_f64(out)
    for b, (n, klen) in enumerate(zip(q_lens, kv_lens)):
        s0 = int(cu[b])
        ref = oracle.attention(q[s0:s0 + n].permute(1, 0, 2)[None], ck[b:b + 1], cv[b:b + 1], pos_offset=klen - n,
                               mask_mode=MASK_CAUSAL, key_lens=[klen], scale=sc)
        assert_close(got[s0:s0 + n], ref[0].transpose(1, 0, 2), "f16", f"seq {b}")


def test_bad_page_entry_zeroes_only_that_sequence():
    q_lens, kv_lens = [40, 60, 30], [300, 200, 100]
    q, kp, vp, table, cu, kl, ck, cv = paged_chunks(q_lens, kv_lens, 4, 2, 64, 32, seed=13)
    table[1, 2] = table.max() + 100       # inside sequence 1's cached positions: reported, rows zeroed
    table[2, 5] = -7                      # past sequence 2's 100 positions (pages 0..3): never read
    sc = scale_of(64)
    out = torch.full((q.shape[0], 4, 64), 5.0, dtype=torch.bfloat16, device=DEV)
    run_paged(q, kp, vp, table, cu, kl, MASK_CAUSAL, 0, sc, out=out)
    assert attn.sync_status() == attn.ATTN_ERR_INVALID_ARG
    assert "page" in attn.last_error()
    assert attn.sync_status() == attn.ATTN_OK
    got = to_numpy_f64(out)
    assert np.all(got[40:100] == 0)
    for b in (0, 2):
        s0, n, klen = int(cu[b]), q_lens[b], kv_lens[b]
        ref = oracle.attention(q[s0:s0 + n].permute(1, 0, 2)[None], ck[b:b + 1], cv[b:b + 1], pos_offset=klen - n,
                               mask_mode=MASK_CAUSAL, key_lens=[klen], scale=sc)
        assert_close(got[s0:s0 + n], ref[0].transpose(1, 0, 2), "bf16", f"seq {b}")


def test_fewer_cached_positions_than_queries_is_reported():
    q_lens, kv_lens = [50, 20], [40, 100]  # sequence 0 has 50 queries but only 40 cached positions
    q, kp, vp, table, cu, kl, ck, cv = paged_chunks(q_lens, kv_lens, 4, 4, 128, 16, seed=14)
    sc = scale_of(128)
    out = torch.full((q.shape[0], 4, 128), 5.0, dtype=torch.bfloat16, device=DEV)
    run_paged(q, kp, vp, table, cu, kl, MASK_CAUSAL, 0, sc, out=out)
    assert attn.sync_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.sync_status() == attn.ATTN_OK
    got = to_numpy_f64(out)
    assert np.all(got[:50] == 0)
    ref = oracle.attention(q[50:70].permute(1, 0, 2)[None], ck[1:2], cv[1:2], pos_offset=80, mask_mode=MASK_CAUSAL,
                           key_lens=[100], scale=sc)
    assert_close(got[50:70], ref[0].transpose(1, 0, 2), "bf16", "seq 1")


def test_bad_cu_seqlens_is_reported_and_not_written():
    q_lens, kv_lens = [30, 30], [30, 60]
    q, kp, vp, table, cu, kl, ck, cv = paged_chunks(q_lens, kv_lens, 4, 2, 64, 16, seed=15)
    cu_bad = cu.clone()
    cu_bad[2] = 61  # past total_q = 60
    out = torch.full((q.shape[0], 4, 64), 5.0, dtype=torch.bfloat16, device=DEV)
    attn.attn_fwd_varlen_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), cu_bad.to(DEV), kl.to(DEV), 31,
                               out=out, scale=0.125)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.sync_status() == attn.ATTN_OK
    assert torch.all(out[30:] == 5.0)                     # sequence 1 is not written
    assert torch.isfinite(out[:30].float()).all() and not torch.all(out[:30] == 5.0)


def test_paged_chunked_prefill_full_size():
    """The timed chunked prefill at its full size: 4 sequences, their newest 512 of 4,096 cached
    positions, 32 query / 8 kv heads, head_dim 128, bf16, causal, 16-row pages in shuffled pool
    order (the TMA page producer).  Every output element is checked against the fp64 oracle, per
    (sequence, head) slab too, and the output equals attn_fwd over the gathered caches bit for
    bit (a causal band starts at key 0, so both split the keys into the same tiles)."""
    from parity_util import assert_close_per_head
    B, Hq, Hkv, D, chunk, kv, ps = 4, 32, 8, 128, 512, 4096, 16
    g = torch.Generator().manual_seed(41)
    caches_k = torch.randn(B, Hkv, kv, D, generator=g).to(torch.bfloat16)
    caches_v = torch.randn(B, Hkv, kv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(B * chunk, Hq, D, generator=g).to(torch.bfloat16)
    max_pages = kv // ps
    table = torch.randperm(B * max_pages, generator=g).view(B, max_pages).to(torch.int32)

    def pool(c):  # pool page table[b, j] holds positions [j ps, (j + 1) ps) of sequence b
        p = torch.empty(B * max_pages, Hkv, ps, D, dtype=torch.bfloat16)
        p[table.flatten().long()] = c.view(B, Hkv, max_pages, ps, D).permute(0, 2, 1, 3, 4).reshape(-1, Hkv, ps, D)
        return p
    cu = torch.arange(0, (B + 1) * chunk, chunk, dtype=torch.int32)
    kl = torch.full((B,), kv, dtype=torch.int32)
    sc = scale_of(D)
    out = run_paged(q, pool(caches_k), pool(caches_v), table, cu, kl, MASK_CAUSAL, 0, sc)
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    qh = q.view(B, chunk, Hq, D).permute(0, 2, 1, 3).contiguous()
    fwd = attn.attn_fwd(qh.to(DEV), caches_k.to(DEV), caches_v.to(DEV), pos_offset=kv - chunk, mask_mode=MASK_CAUSAL,
                        scale=sc)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    got = out.view(B, chunk, Hq, D).permute(0, 2, 1, 3)
    assert torch.equal(got.cpu(), fwd.cpu())
    ref = oracle.attention(qh, caches_k, caches_v, pos_offset=kv - chunk, mask_mode=MASK_CAUSAL, scale=sc)
    assert_close_per_head(to_numpy_f64(got), ref, "bf16", "paged chunked prefill, full size")


@pytest.mark.parametrize("page_size", [16, 32, 7])
def test_paged_chunks_many_ragged_sequences(page_size):
    """Forty sequences with random chunk lengths (0 to 200 queries, some a whole prefill) and
    0 to 600 older cached positions, 8 query / 2 kv heads, head_dim 128, causal with and without
    a window: every sequence against the oracle."""
    rng = np.random.default_rng(100 + page_size)
    n = 40
    q_lens = [int(x) for x in rng.integers(0, 201, n)]
    q_lens[0], q_lens[1] = 0, 1
    kv_lens = [ql + int(x) for ql, x in zip(q_lens, rng.integers(0, 601, n))]
    kv_lens[2] = q_lens[2]  # a whole prefill: no older positions
    for mode, window in ((MASK_CAUSAL, 0), (MASK_CAUSAL_WINDOW, 97)):
        q, kp, vp, table, cu, kl, ck, cv = paged_chunks(q_lens, kv_lens, 8, 2, 128, page_size,
                                                        seed=200 + page_size + mode)
        sc = scale_of(128)
        got = to_numpy_f64(run_paged(q, kp, vp, table, cu, kl, mode, window, sc))
        assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
        for b, (m, klen) in enumerate(zip(q_lens, kv_lens)):
            if m == 0:
                continue
            s0 = int(cu[b])
            ref = oracle.attention(q[s0:s0 + m].permute(1, 0, 2)[None], ck[b:b + 1], cv[b:b + 1], pos_offset=klen - m,
                                   mask_mode=mode, window=window, key_lens=[klen], scale=sc)
            assert_close(got[s0:s0 + m], ref[0].transpose(1, 0, 2), "bf16", f"seq {b} (len {m}, kv {klen}), mode {mode}")
