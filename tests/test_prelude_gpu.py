"""GPU parity of the attention prelude (attn_qkv_prelude) against the fp64 oracle.

Each output element is one fp32 computation rounded once to the output type, so the
bound is elementwise: |got - ref| <= 2^-8 |ref| (bf16) or 2^-10 |ref| (fp16), plus 1e-5
for the fp32 arithmetic (norm, rotation) before the rounding."""
import numpy as np
import pytest
import torch

import head_attention_attn_gb300 as attn
from oracle import prelude as P

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from head_attention_attn_gb300 import build
    build.build_library()
    attn.load()
    yield
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()


def rope_tables(positions, hd, base=1.0e6):
    j = torch.arange(hd // 2, dtype=torch.float64)
    ang = torch.arange(positions, dtype=torch.float64)[:, None] * base ** (-2.0 * j / hd)[None, :]
    return torch.cos(ang).float(), torch.sin(ang).float()


def assert_elementwise(got, ref, dtype, what):
    got = got.double().cpu().numpy()
    rel = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -10
    excess = np.abs(got - ref) - rel * np.abs(ref)
    assert np.all(np.isfinite(got)), what
    assert excess.max() <= 1e-5, f"{what}: worst excess {excess.max():.3e}"


def inputs(T, Hq, Hkv, hd, dtype, seed, positions):
    g = torch.Generator().manual_seed(seed)
    qkv = (torch.randn(T, (Hq + 2 * Hkv) * hd, generator=g) * 2.0).to(dtype)
    qw = torch.rand(hd, generator=g) + 0.5
    kw = torch.rand(hd, generator=g) + 0.5
    cos, sin = rope_tables(positions, hd)
    return qkv, qw, kw, cos, sin


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_prelude_matches_oracle(dtype, hd, mode):
    T, Hq, Hkv, pos = 37, 4, 2, 5
    qkv, qw, kw, cos, sin = inputs(T, Hq, Hkv, hd, dtype, seed=9000 + hd + mode, positions=64)
    q, k, v = attn.attn_qkv_prelude(qkv.to(DEV), Hq, Hkv, hd, qk_mode=mode, cos=cos.to(DEV), sin=sin.to(DEV),
                                    q_norm_w=qw.to(DEV), k_norm_w=kw.to(DEV), pos_offset=pos, eps=1e-6)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    rq, rk, rv = P.split_qkv_norm_rope(qkv, qw, kw, cos, sin, q_heads=Hq, kv_heads=Hkv, head_dim=hd, pos_offset=pos,
                                       eps=1e-6, qk_mode=mode)
    assert_elementwise(q, rq, dtype, f"q mode {mode}")
    assert_elementwise(k, rk, dtype, f"k mode {mode}")
    assert torch.equal(v.cpu(), torch.from_numpy(rv).to(dtype))  # V is a plain copy


@pytest.mark.parametrize("mode", [1, 3])
def test_prelude_into_cache_writes_only_its_slot(mode):
    T, Hq, Hkv, hd, cap, start = 29, 8, 2, 128, 100, 40
    qkv, qw, kw, cos, sin = inputs(T, Hq, Hkv, hd, torch.bfloat16, seed=9100 + mode, positions=128)
    kc = torch.full((Hkv, cap, hd), 3.0, dtype=torch.bfloat16, device=DEV)
    vc = torch.full((Hkv, cap, hd), -2.0, dtype=torch.bfloat16, device=DEV)
    q, k2, v2 = attn.attn_qkv_prelude(qkv.to(DEV), Hq, Hkv, hd, qk_mode=mode, cos=cos.to(DEV), sin=sin.to(DEV),
                                      q_norm_w=qw.to(DEV), k_norm_w=kw.to(DEV), pos_offset=start, eps=1e-6,
                                      k_cache=kc, v_cache=vc, cache_len=start)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert k2.data_ptr() == kc.data_ptr()
    rq, rkc, rvc = P.split_qkv_norm_rope_into_cache(qkv, qw, kw, cos, sin, kc.cpu(), vc.cpu(), q_heads=Hq,
                                                    kv_heads=Hkv, head_dim=hd, pos_offset=start, eps=1e-6,
                                                    qk_mode=mode, cache_len=start)
    assert_elementwise(q, rq, torch.bfloat16, "q")
    assert_elementwise(kc, rkc, torch.bfloat16, "k cache")
    assert torch.equal(vc.cpu(), torch.from_numpy(rvc).to(torch.bfloat16))
    keep = torch.ones(cap, dtype=torch.bool)
    keep[start:start + T] = False
    assert torch.all(kc[:, keep] == 3.0) and torch.all(vc[:, keep] == -2.0)


def test_prelude_full_size_qwen_like():
    """4 sequences x 4096 tokens of a 32q/8kv, head_dim 128 layer with QK-norm."""
    T, Hq, Hkv, hd = 16384, 32, 8, 128
    qkv, qw, kw, cos, sin = inputs(T, Hq, Hkv, hd, torch.bfloat16, seed=9200, positions=T)
    q, k, v = attn.attn_qkv_prelude(qkv.to(DEV), Hq, Hkv, hd, qk_mode=1, cos=cos.to(DEV), sin=sin.to(DEV),
                                    q_norm_w=qw.to(DEV), k_norm_w=kw.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    rows = np.r_[0:3, 4095:4098, T - 3:T]  # token rows at the edges of the table and the buffer
    rq, rk, rv = [], [], []  # one oracle call per row, at that row's position
    for r in rows:
        a, b, c = P.split_qkv_norm_rope(qkv[r:r + 1], qw, kw, cos, sin, q_heads=Hq, kv_heads=Hkv, head_dim=hd,
                                        pos_offset=int(r), eps=1e-6, qk_mode=1)
        rq.append(a[:, 0]), rk.append(b[:, 0]), rv.append(c[:, 0])
    assert_elementwise(q[:, rows].permute(1, 0, 2), np.stack(rq), torch.bfloat16, "q")
    assert_elementwise(k[:, rows].permute(1, 0, 2), np.stack(rk), torch.bfloat16, "k")
    assert torch.equal(v[:, rows].permute(1, 0, 2).cpu(), torch.from_numpy(np.stack(rv)).to(torch.bfloat16))


def test_prelude_feeds_attention():
    """Prelude output goes straight into attn_fwd (head-major), as the pages chain them."""
    T, Hq, Hkv, hd = 300, 8, 2, 128
    qkv, qw, kw, cos, sin = inputs(T, Hq, Hkv, hd, torch.bfloat16, seed=9300, positions=T)
    q, k, v = attn.attn_qkv_prelude(qkv.to(DEV), Hq, Hkv, hd, qk_mode=2, cos=cos.to(DEV), sin=sin.to(DEV))
    out = attn.attn_fwd(q[None], k[None], v[None], mask_mode=attn.MASK_CAUSAL)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("mode", [1, 3])
def test_decode_step_prelude_then_attention(mode):
    """One decode step for 5 items with their own caches: the per-item prelude appends each
    item's K/V at its cache length and writes its Q, then attn_decode_caches attends over
    the grown caches.  Both against the oracles (prelude oracle, then attention oracle)."""
    import oracle
    m, Hq, Hkv, hd, cap = 5, 8, 2, 128, 300
    lens = [0, 17, 128, 250, 299]
    g = torch.Generator().manual_seed(9400 + mode)
    # N(0, 1) like every attention input here: the bf16 output bound (1e-2) assumes |o| <~ 5
    qkv = torch.randn(m, (Hq + 2 * Hkv) * hd, generator=g).to(torch.bfloat16)
    qw, kw = torch.rand(hd, generator=g) + 0.5, torch.rand(hd, generator=g) + 0.5
    cos, sin = rope_tables(cap, hd)
    ks = [torch.randn(Hkv, cap, hd, generator=g).to(torch.bfloat16) for _ in range(m)]
    vs = [torch.randn(Hkv, cap, hd, generator=g).to(torch.bfloat16) for _ in range(m)]
    kd, vd = [k.to(DEV) for k in ks], [v.to(DEV) for v in vs]
    cl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    q = attn.attn_qkv_prelude_caches(qkv.to(DEV), kd, vd, cl, Hq, Hkv, hd, qk_mode=mode, cos=cos.to(DEV),
                                     sin=sin.to(DEV), q_norm_w=qw.to(DEV), k_norm_w=kw.to(DEV), eps=1e-6)
    out = attn.attn_decode_caches(q, kd, vd, cl + 1)
    torch.cuda.synchronize()
    assert attn.sync_status() == attn.ATTN_OK, attn.last_error()
    for i in range(m):
        rq, rk, rv = P.split_qkv_norm_rope(qkv[i:i + 1], qw, kw, cos, sin, q_heads=Hq, kv_heads=Hkv, head_dim=hd,
                                           pos_offset=lens[i], eps=1e-6, qk_mode=mode)
        assert_elementwise(q[i], rq[:, 0], torch.bfloat16, f"q item {i}")
        assert_elementwise(kd[i][:, lens[i]], rk[:, 0], torch.bfloat16, f"k item {i}")
        assert torch.equal(vd[i][:, lens[i]].cpu(), torch.from_numpy(rv[:, 0]).to(torch.bfloat16))
        keep = torch.ones(cap, dtype=torch.bool)
        keep[lens[i]] = False
        assert torch.equal(kd[i][:, keep].cpu(), ks[i][:, keep]) and torch.equal(vd[i][:, keep].cpu(), vs[i][:, keep])
        n = lens[i] + 1
        ref = oracle.attention(q[i].cpu()[None, :, None, :], kd[i].cpu()[None], vd[i].cpu()[None], pos_offset=n - 1,
                               mask_mode=attn.MASK_CAUSAL, key_lens=[n],
                               scale=float(torch.tensor(1.0 / hd ** 0.5, dtype=torch.float32)))
        from parity_util import assert_close
        assert_close(out[i].double().cpu().numpy(), ref[0, :, 0, :], "bf16", f"decode item {i}")


def test_prelude_caches_bad_items_are_reported_not_written():
    m, Hq, Hkv, hd, cap = 3, 4, 2, 64, 16
    g = torch.Generator().manual_seed(9500)
    qkv = torch.randn(m, (Hq + 2 * Hkv) * hd, generator=g).to(torch.bfloat16).to(DEV)
    kd = [torch.zeros(Hkv, cap, hd, dtype=torch.bfloat16, device=DEV) for _ in range(m)]
    vd = [torch.zeros(Hkv, cap, hd, dtype=torch.bfloat16, device=DEV) for _ in range(m)]
    cl = torch.tensor([3, cap, -1], dtype=torch.int32, device=DEV)  # items 1 and 2 are out of range
    q = torch.full((m, Hq, hd), 9.0, dtype=torch.bfloat16, device=DEV)
    attn.attn_qkv_prelude_caches(qkv, kd, vd, cl, Hq, Hkv, hd, qk_mode=attn.QK_COPY, q_out=q)
    assert attn.sync_status() == attn.ATTN_ERR_INVALID_ARG
    assert attn.sync_status() == attn.ATTN_OK
    assert torch.all(kd[1] == 0) and torch.all(kd[2] == 0) and torch.all(q[1:] == 9.0)
    assert torch.equal(q[0], qkv[0, :Hq * hd].view(Hq, hd))  # item 0 went through (copy mode)
