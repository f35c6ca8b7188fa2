"""Pins of the fp64 prelude oracle (oracle/prelude.py) to things other than itself:
complex-number rotation, torch's RMS norm, closed forms, invariants and one-hot routing.
A set of planted mistakes (sign, pairing, order, scale, routing) must each fail a pin."""
import numpy as np
import pytest
import torch

from oracle import prelude as P

RNG = np.random.default_rng(1234)


def tables(positions, hd, base=10000.0):
    j = np.arange(hd // 2)
    ang = np.arange(positions)[:, None] * base ** (-2.0 * j / hd)[None, :]
    return np.cos(ang), np.sin(ang)


def run(impl, qkv, qw, kw, cos, sin, Hq, Hkv, hd, pos, eps, mode):
    return impl(qkv, qw, kw, cos, sin, q_heads=Hq, kv_heads=Hkv, head_dim=hd, pos_offset=pos, eps=eps, qk_mode=mode)


def pin_failures(impl):
    """Run every pin against `impl` (a split_qkv_norm_rope implementation); return failures."""
    fails = []
    Hq, Hkv, hd, T = 4, 2, 16, 5
    qkv = RNG.standard_normal((T, (Hq + 2 * Hkv) * hd))
    qw, kw = RNG.uniform(0.5, 1.5, hd), RNG.uniform(0.5, 1.5, hd)
    cos, sin = tables(64, hd)
    q_in = qkv[:, :Hq * hd].reshape(T, Hq, hd)
    k_in = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(T, Hkv, hd)
    v_in = qkv[:, (Hq + Hkv) * hd:].reshape(T, Hkv, hd)

    def check(name, cond):
        if not cond:
            fails.append(name)

    # 1. mode 0 is a plain split + transpose (one-hot routing of every feature)
    q, k, v = run(impl, qkv, qw, kw, cos, sin, Hq, Hkv, hd, 3, 1e-6, 0)
    check("transpose-q", np.array_equal(q, q_in.transpose(1, 0, 2)))
    check("transpose-k", np.array_equal(k, k_in.transpose(1, 0, 2)))
    check("transpose-v", np.array_equal(v, v_in.transpose(1, 0, 2)))

    # 2. RoPE at position 0 (cos 1, sin 0) is the identity, for both pairings
    for mode in (2, 3):
        q, k, v = run(impl, qkv[:1], qw, kw, cos, sin, Hq, Hkv, hd, 0, 1e-6, mode)
        check(f"pos0-identity-{mode}", np.allclose(q[:, 0], q_in[0], atol=0) and np.allclose(k[:, 0], k_in[0], atol=0))

    # 3. half-split rotation == complex multiplication z_j * e^{i angle_j}, z_j = x_j + i x_{j+hd/2}
    pos = 7
    q, k, v = run(impl, qkv, qw, kw, cos, sin, Hq, Hkv, hd, pos, 1e-6, 2)
    ang = np.arctan2(sin[pos:pos + T], cos[pos:pos + T])[:, None, :]
    z = (q_in[..., :hd // 2] + 1j * q_in[..., hd // 2:]) * np.exp(1j * ang)
    ref = np.concatenate([z.real, z.imag], axis=-1).transpose(1, 0, 2)
    check("complex-half-split", np.allclose(q, ref, atol=1e-12))
    check("v-untouched-by-rope", np.array_equal(v, v_in.transpose(1, 0, 2)))

    # 4. interleaved rotation == complex multiplication with z_j = x_{2j} + i x_{2j+1}
    q, k, v = run(impl, qkv, qw, kw, cos, sin, Hq, Hkv, hd, pos, 1e-6, 3)
    z = (k_in[..., 0::2] + 1j * k_in[..., 1::2]) * np.exp(1j * ang)
    ref = np.empty_like(k_in)
    ref[..., 0::2], ref[..., 1::2] = z.real, z.imag
    check("complex-interleaved", np.allclose(k, ref.transpose(1, 0, 2), atol=1e-12))

    # 5. a quarter turn (cos 0, sin 1): half-split (a, b) -> (-b, a)
    c90, s90 = np.zeros((1, hd // 2)), np.ones((1, hd // 2))
    q, k, v = run(impl, qkv[:1], qw, kw, c90, s90, Hq, Hkv, hd, 0, 1e-6, 2)
    a, b = q_in[0][:, :hd // 2], q_in[0][:, hd // 2:]
    check("quarter-turn", np.array_equal(q[:, 0], np.concatenate([-b, a], axis=-1)))

    # 6. rotation keeps every row's length; rotating by x then y equals rotating by x + y
    q, k, v = run(impl, qkv, qw, kw, cos, sin, Hq, Hkv, hd, 11, 1e-6, 2)
    check("norm-preserved", np.allclose(np.linalg.norm(q, axis=-1), np.linalg.norm(q_in, axis=-1).T, rtol=1e-12))
    c2, s2 = tables(64, hd)
    once = run(impl, qkv[:1], qw, kw, c2, s2, Hq, Hkv, hd, 9, 1e-6, 2)[0][:, 0]
    first = run(impl, qkv[:1], qw, kw, c2, s2, Hq, Hkv, hd, 4, 1e-6, 2)[0][:, 0]
    re = np.concatenate([first.reshape(1, Hq * hd), qkv[:1, Hq * hd:]], axis=1)
    twice = run(impl, re, qw, kw, c2, s2, Hq, Hkv, hd, 5, 1e-6, 2)[0][:, 0]
    check("angle-addition", np.allclose(once, twice, atol=1e-12))

    # 7. mode 1 = torch RMS norm (fp64) then the half-split rotation, per head, Q and K
    q, k, v = run(impl, qkv, qw, kw, cos, sin, Hq, Hkv, hd, pos, 1e-5, 1)
    qn = torch.nn.functional.rms_norm(torch.from_numpy(q_in), (hd,), torch.from_numpy(qw), eps=1e-5).numpy()
    z = (qn[..., :hd // 2] + 1j * qn[..., hd // 2:]) * np.exp(1j * ang)
    ref = np.concatenate([z.real, z.imag], axis=-1).transpose(1, 0, 2)
    check("norm-then-rope-q", np.allclose(q, ref, atol=1e-12))
    kn = torch.nn.functional.rms_norm(torch.from_numpy(k_in), (hd,), torch.from_numpy(kw), eps=1e-5).numpy()
    z = (kn[..., :hd // 2] + 1j * kn[..., hd // 2:]) * np.exp(1j * ang)
    ref = np.concatenate([z.real, z.imag], axis=-1).transpose(1, 0, 2)
    check("norm-then-rope-k", np.allclose(k, ref, atol=1e-12))

    # 8. RMS norm closed form: a constant row c with eps 0 gives sign(c) * w
    const = np.full((1, (Hq + 2 * Hkv) * hd), -3.0)
    q, k, v = run(impl, const, qw, kw, np.ones((1, hd // 2)), np.zeros((1, hd // 2)), Hq, Hkv, hd, 0, 0.0, 1)
    check("norm-constant-row", np.allclose(q[:, 0], -qw[None, :], atol=1e-15) and np.allclose(k[:, 0], -kw, atol=1e-15))
    return fails


def test_oracle_passes_every_pin():
    assert pin_failures(P.split_qkv_norm_rope) == []


# ---------------------------------------------------------------------------- planted mistakes

def _mutant(kind):
    def impl(qkv, qw, kw, cos, sin, *, q_heads, kv_heads, head_dim, pos_offset, eps, qk_mode):
        x = np.asarray(qkv, dtype=np.float64)
        T, hd = x.shape[0], head_dim
        q = x[:, :q_heads * hd].reshape(T, q_heads, hd)
        k = x[:, q_heads * hd:(q_heads + kv_heads) * hd].reshape(T, kv_heads, hd)
        v = x[:, (q_heads + kv_heads) * hd:].reshape(T, kv_heads, hd)
        if kind == "k-from-v":
            k = v
        if qk_mode == 1:
            e = 0.0 if kind == "no-eps-and-mean-as-sum" else eps
            den = np.sum if kind == "no-eps-and-mean-as-sum" else np.mean
            q = q / np.sqrt(den(q * q, axis=-1, keepdims=True) + e) * qw
            k = k / np.sqrt(den(k * k, axis=-1, keepdims=True) + e) * (qw if kind == "q-weight-on-k" else kw)
        if qk_mode in (1, 2, 3):
            off = pos_offset + (1 if kind == "position-off-by-one" else 0)
            c = np.asarray(cos)[off:off + T][:, None, :]
            s = np.asarray(sin)[off:off + T][:, None, :]
            if kind == "sign-flip":
                s = -s
            if kind == "adjacent-pairs-for-half-split" or qk_mode == 3:
                rot = P.rope_interleaved
            else:
                rot = P.rope_half_split
            q = rot(q, c, s)
            k = rot(k, c, s)
            if kind == "rope-on-v":
                v = rot(v, c, s)
        if kind == "norm-after-rope" and qk_mode == 1:
            q = P.rms_norm(P.rope_half_split(x[:, :q_heads * hd].reshape(T, q_heads, hd),
                                             np.asarray(cos)[pos_offset:pos_offset + T][:, None, :],
                                             np.asarray(sin)[pos_offset:pos_offset + T][:, None, :]), qw, eps)
        if kind == "token-major-out":
            return q.reshape(q.shape[1], q.shape[0], hd), k.transpose(1, 0, 2), v.transpose(1, 0, 2)
        return q.transpose(1, 0, 2), k.transpose(1, 0, 2), v.transpose(1, 0, 2)
    return impl


@pytest.mark.parametrize("kind", ["sign-flip", "adjacent-pairs-for-half-split", "norm-after-rope", "rope-on-v",
                                  "no-eps-and-mean-as-sum", "q-weight-on-k", "position-off-by-one", "k-from-v",
                                  "token-major-out"])
def test_planted_mistake_fails_a_pin(kind):
    try:
        fails = pin_failures(_mutant(kind))
    except (IndexError, ValueError) as e:  # a mutant that cannot even run the pins is caught too
        fails = [f"raised {type(e).__name__}"]
    assert fails, f"mutant {kind} passed every pin"


def test_unmutated_copy_of_the_mutant_harness_passes():
    # the harness itself is a faithful second implementation when no mistake is planted
    assert pin_failures(_mutant("none")) == []


def test_into_cache_writes_only_its_slot():
    Hq, Hkv, hd, T, cap, start = 2, 2, 8, 3, 10, 4
    qkv = RNG.standard_normal((T, (Hq + 2 * Hkv) * hd))
    cos, sin = tables(16, hd)
    ck0, cv0 = RNG.standard_normal((Hkv, cap, hd)), RNG.standard_normal((Hkv, cap, hd))
    q, ck, cv = P.split_qkv_norm_rope_into_cache(qkv, np.ones(hd), np.ones(hd), cos, sin, ck0, cv0, q_heads=Hq,
                                                 kv_heads=Hkv, head_dim=hd, pos_offset=5, eps=1e-6, qk_mode=2,
                                                 cache_len=start)
    q2, k2, v2 = P.split_qkv_norm_rope(qkv, np.ones(hd), np.ones(hd), cos, sin, q_heads=Hq, kv_heads=Hkv, head_dim=hd,
                                       pos_offset=5, eps=1e-6, qk_mode=2)
    assert np.array_equal(q, q2)
    assert np.array_equal(ck[:, start:start + T], k2) and np.array_equal(cv[:, start:start + T], v2)
    keep = np.ones(cap, bool)
    keep[start:start + T] = False
    assert np.array_equal(ck[:, keep], ck0[:, keep]) and np.array_equal(cv[:, keep], cv0[:, keep])
    with pytest.raises(ValueError):
        P.split_qkv_norm_rope_into_cache(qkv, np.ones(hd), np.ones(hd), cos, sin, ck0, cv0, q_heads=Hq, kv_heads=Hkv,
                                         head_dim=hd, pos_offset=5, eps=1e-6, qk_mode=2, cache_len=8)
