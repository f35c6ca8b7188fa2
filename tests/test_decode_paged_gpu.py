"""Decode over paged KV caches (attn_decode_paged) on the GPU.

Item i's cache is cut into pages of page_size positions, [Hkv, page_size, D] each, held in
two pools [num_pages, Hkv, page_size, D] and addressed by page_table[i][j] for positions
j*page_size .. (j+1)*page_size - 1.  Gathering item i's pages back into one [Hkv, capacity, D]
cache and running attn_decode_caches over it computes the same numbers in the same order, so
the two agree bit for bit; the gathered caches are also checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
import oracle
from head_attention_attn_gb300.inputs import MASK_CAUSAL, MASK_CAUSAL_WINDOW
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


def paged_case(m, Hq, Hkv, D, page_size, max_pages, num_pages, lens, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(m, Hq, D, generator=g).to(dtype)
    k_pool = torch.randn(num_pages, Hkv, page_size, D, generator=g).to(dtype)
    v_pool = torch.randn(num_pages, Hkv, page_size, D, generator=g).to(dtype)
    # a random page table (pages may repeat across and within items)
    table = torch.randint(0, num_pages, (m, max_pages), generator=g, dtype=torch.int32)
    return q, k_pool, v_pool, table, torch.tensor(lens, dtype=torch.int32)


def gathered(pool, table):
    """[m, Hkv, max_pages * page_size, D] per-item caches assembled from the pool pages."""
    m, max_pages = table.shape
    _, Hkv, ps, D = pool.shape
    x = pool[table.long()]                      # [m, max_pages, Hkv, ps, D]
    return x.permute(0, 2, 1, 3, 4).reshape(m, Hkv, max_pages * ps, D).contiguous()


def reference(q, kc, vc, lens, window, scale):
    rows = []
    for i in range(q.shape[0]):
        n = int(min(max(int(lens[i]), 0), kc.shape[2]))
        if n == 0:
            rows.append(np.zeros((q.shape[1], q.shape[2])))
            continue
        mode = MASK_CAUSAL_WINDOW if window > 0 else MASK_CAUSAL
        r = oracle.attention(q[i][None, :, None, :], kc[i][None], vc[i][None], pos_offset=n - 1, mask_mode=mode,
                             window=window, key_lens=[n], scale=scale)
        rows.append(r[0, :, 0, :])
    return np.stack(rows)


def run_both(q, k_pool, v_pool, table, kl, window):
    scale = float(torch.tensor(1.0 / q.shape[2] ** 0.5, dtype=torch.float32))
    qd, kp, vp, td, kld = q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), table.to(DEV), kl.to(DEV)
    paged = attn.attn_decode_paged(qd, kp, vp, td, kld, sliding_window=window, scale=scale)
    kc, vc = gathered(kp, td), gathered(vp, td)
    cont = attn.attn_decode_caches(qd, list(kc), list(vc), kld, sliding_window=window, scale=scale)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    return paged, cont, kc.cpu(), vc.cpu(), scale


def tma_page(page_size):
    """Page sizes the tensor-core decode copies by TMA: whole pages of 8 to 128 rows dividing 128,
    or multiples of 128 rows."""
    return (8 <= page_size <= 128 and 128 % page_size == 0) or page_size % 128 == 0


def paged_on_tensor_cores(G, page_size):
    """The faster kernel for paged caches at head_dim 128, as measured: the tensor-core decode at
    4 query heads per kv head when TMA copies pages of 32 rows or more, at 8 when TMA can copy the
    pages or they are shorter than 4 rows (gathered); the CUDA-core decode otherwise."""
    if G == 4:
        return tma_page(page_size) and page_size >= 32
    return G == 8 and (tma_page(page_size) or page_size < 4)


def same_kernel(D, G, page_size):
    """Paged and per-item caches run the same kernel, and then agree bit for bit: the CUDA-core
    decode for both, or the tensor-core decode for both (per-item caches at groups 4 and 8, by TMA
    through a tensor map per item cache, into the same tiles as the paged pages)."""
    if D != 128 or G in (1, 2):
        return True
    caches_tc = G in (4, 8)
    return caches_tc == paged_on_tensor_cores(G, page_size)


@pytest.mark.parametrize("D,G", [(128, 4), (128, 8), (128, 1), (64, 8), (64, 2)])
@pytest.mark.parametrize("page_size,window", [(16, 0), (48, 300), (100, 0), (1, 0), (2048, 64), (32, 0), (8, 77)])
def test_paged_equals_gathered_caches(D, G, page_size, window):
    Hkv, m = 2, 4
    max_pages = max(1, 1500 // page_size) if page_size > 1 else 300
    cap = max_pages * page_size
    lens = [1, cap // 3, cap, cap + 500]  # the last clamps to the capacity
    q, kp, vp, table, kl = paged_case(m, G * Hkv, Hkv, D, page_size, max_pages, 2 * max_pages + 3, lens,
                                      seed=31 * D + G + page_size + window)
    paged, cont, kc, vc, scale = run_both(q, kp, vp, table, kl, window)
    if same_kernel(D, G, page_size):
        assert torch.equal(paged, cont)
    ref = reference(q, kc, vc, kl, window, scale)
    assert_close(paged.double().cpu().numpy(), ref, "bf16", f"paged D={D} G={G} ps={page_size} w={window}")
    assert_close(cont.double().cpu().numpy(), ref, "bf16", f"gathered D={D} G={G} ps={page_size} w={window}")


@pytest.mark.parametrize("window", [0, 200])
def test_paged_f16_against_oracle(window):
    q, kp, vp, table, kl = paged_case(3, 8, 2, 128, 64, 20, 50, [1000, 17, 1280], seed=77, dtype=torch.float16)
    paged, cont, kc, vc, scale = run_both(q, kp, vp, table, kl, window)
    ref = reference(q, kc, vc, kl, window, scale)
    assert_close(paged.double().cpu().numpy(), ref, "f16", "paged f16")
    assert_close(cont.double().cpu().numpy(), ref, "f16", "gathered f16")


@pytest.mark.parametrize("Hq,D", [(4, 64), (8, 128)])  # the CUDA-core and the tensor-core decode
def test_bad_page_entry_is_reported_and_that_item_zeroed(Hq, D):
    q, kp, vp, table, kl = paged_case(3, Hq, 2, D, 32, 8, 10, [200, 200, 200], seed=78)
    table[1, 3] = 10  # one past the pool: item 1 sees positions up to 199, page 3 is visible
    table[2, 7] = -1  # outside item 2's visible positions (pages 0..6): never read, no error
    scale = float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))
    out = attn.attn_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), kl.to(DEV), scale=scale)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_ERR_INVALID_ARG
    assert "page" in attn.last_error()
    assert attn.sync_status() == attn.ATTN_OK
    assert torch.all(out[1] == 0)
    good = table.clone()
    good[1, 3] = 0
    kc, vc = gathered(kp, good), gathered(vp, good)
    ref = reference(q, kc, vc, kl, 0, scale)
    assert_close(out[[0, 2]].double().cpu().numpy(), ref[[0, 2]], "bf16", "paged, good items")


def test_zero_lengths_give_zeros():
    q, kp, vp, table, kl = paged_case(2, 4, 4, 128, 16, 4, 4, [0, 0], seed=79)
    out = torch.full_like(q, 3.0).to(DEV)
    attn.attn_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), kl.to(DEV), out)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.all(out == 0)


def test_zero_capacity_zero_fills():
    q, kp, vp, _, kl = paged_case(2, 4, 4, 128, 16, 4, 4, [5, 9], seed=80)
    table = torch.zeros((2, 0), dtype=torch.int32, device=DEV)  # max_pages 0
    out = torch.full_like(q, 3.0).to(DEV)
    attn.attn_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table, kl.to(DEV), out)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.all(out == 0)


@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("page_size", [16, 8, 32, 128, 256, 2])
def test_tensor_core_paged_decode_splits(G, page_size):
    """Few items with long caches: the tensor-core decode splits each item's keys over a
    cluster; paged and gathered caches still agree bit for bit and match the oracle."""
    Hkv, m, D = 2, 2, 128
    max_pages = 6000 // page_size
    cap = max_pages * page_size
    q, kp, vp, table, kl = paged_case(m, G * Hkv, Hkv, D, page_size, max_pages, max_pages + 7, [cap, cap - 1234],
                                      seed=90 + G + page_size)
    paged, cont, kc, vc, scale = run_both(q, kp, vp, table, kl, 0)
    if same_kernel(D, G, page_size):
        assert torch.equal(paged, cont)
    ref = reference(q, kc, vc, kl, 0, scale)
    assert_close(paged.double().cpu().numpy(), ref, "bf16", f"paged splits G={G} ps={page_size}")
    assert_close(cont.double().cpu().numpy(), ref, "bf16", f"gathered splits G={G} ps={page_size}")


@pytest.mark.parametrize("G", [4, 8])
def test_decode_forms_full_size(G):
    """The decode legs the bench times, at their full size: 64 items of 8,192 cached positions,
    8 kv heads, head_dim 128, bf16, 4 or 8 query heads per kv head.  The same caches go in
    contiguous (attn_fwd), per item (attn_decode_caches) and in 16- and 128-row pages in shuffled
    pool order (attn_decode_paged).  Forms that run the same kernel as the contiguous decode
    agree with it bit for bit; every form is checked against the oracle on sampled (item, head)
    rows (the contiguous decode is compared on every row by its own full-size test)."""
    m, Hkv, cap, D = 64, 8, 8192, 128
    Hq = G * Hkv
    gen = torch.Generator(device=DEV).manual_seed(50 + G)
    k = torch.randn(m, Hkv, cap, D, generator=gen, device=DEV, dtype=torch.bfloat16)
    v = torch.randn(m, Hkv, cap, D, generator=gen, device=DEV, dtype=torch.bfloat16)
    q = torch.randn(m, Hq, D, generator=gen, device=DEV, dtype=torch.bfloat16)
    kl = torch.full((m,), cap, dtype=torch.int32, device=DEV)
    scale = float(torch.tensor(1.0 / D ** 0.5, dtype=torch.float32))
    cont = attn.attn_fwd(q.view(m, Hq, 1, D), k, v, pos_offset=cap - 1, mask_mode=MASK_CAUSAL, scale=scale)[:, :, 0]
    per_item = attn.attn_decode_caches(q, list(k), list(v), kl, scale=scale)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.equal(per_item, cont)  # the tensor-core decode for both, the same tiles
    forms = {"contiguous": cont, "per-item caches": per_item}
    g = torch.Generator().manual_seed(60 + G)
    for ps in (16, 128):
        pages = cap // ps
        table = torch.randperm(m * pages, generator=g).view(m, pages).to(torch.int32).to(DEV)

        def pool(c):
            p = torch.empty(m * pages, Hkv, ps, D, dtype=torch.bfloat16, device=DEV)
            p[table.flatten().long()] = c.view(m, Hkv, pages, ps, D).permute(0, 2, 1, 3, 4).reshape(-1, Hkv, ps, D)
            return p
        paged = attn.attn_decode_paged(q, pool(k), pool(v), table, kl, scale=scale)
        torch.cuda.synchronize()
        assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
        if paged_on_tensor_cores(G, ps):
            assert torch.equal(paged, cont), f"page {ps}"
        forms[f"paged {ps}"] = paged
    rng = np.random.default_rng(70 + G)
    picks = sorted({(0, 0), (0, Hq - 1), (m - 1, 0), (m - 1, Hq - 1)} |
                   {(int(rng.integers(m)), int(rng.integers(Hq))) for _ in range(40)})
    ref = np.stack([oracle.attention(q[b, h].cpu()[None, None, None], k[b:b + 1, h // G:h // G + 1].cpu(),
                                     v[b:b + 1, h // G:h // G + 1].cpu(), pos_offset=cap - 1, mask_mode=MASK_CAUSAL,
                                     scale=scale)[0, 0, 0] for b, h in picks])
    for name, out in forms.items():
        got = np.stack([out[b, h].double().cpu().numpy() for b, h in picks])
        assert_close(got, ref, "bf16", f"{name}, G={G}, {len(picks)} sampled rows")
