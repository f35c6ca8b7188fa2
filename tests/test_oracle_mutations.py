"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle/attn_oracle.c, applies one plausible slip (an
off-by-one in a mask, a dropped scale, a wrong head mapping, a transposed
operand, a skipped normalisation...), builds it with gcc on the CPU and runs a
quick battery of the pins against that build.  The unmodified source must pass
the battery and every mutant must fail it.
"""
import json
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "attn_oracle.c")

MUTATIONS = {
    "causal_off_by_one": ("return j <= qpos;", "return j < qpos;"),
    "window_half_rounds_up": ("d <= (long long)(window / 2)", "d <= (long long)((window + 1) / 2)"),
    "causal_window_inclusive_edge": ("return j > qpos - (long long)window;",
                                     "return j >= qpos - (long long)window;"),
    "scale_dropped": ("s[j] = jb->scale * acc;", "s[j] = acc;"),
    "gqa_interleaved_heads": ("const int hk = hq / group;", "const int hk = hq % jb->Hkv;"),
    "key_padding_ignored": ("allowed[j] = (unsigned char)(j < klen && ",
                            "allowed[j] = (unsigned char)(j < Lk && "),
    "v_read_as_k": ("const float *vrow = vh + j * D;", "const float *vrow = kh + j * D;"),
    "no_normalisation": ("for (long long j = 0; j < Lk; ++j) s[j] /= sum;",
                         "for (long long j = 0; j < Lk; ++j) s[j] /= 1.0;"),
    "pos_offset_ignored": ("const long long qpos = (long long)jb->P + i;",
                           "const long long qpos = i;"),
    "query_row_transposed": ("const float *qrow = jb->q + row * (long long)D;",
                             "const float *qrow = jb->q + ((row % jb->Lq) * (jb->B * jb->Hq) + (row / jb->Lq)) * (long long)D;"),
}


def _build(tmp_path, text, name):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(src), "-lm", "-lpthread"], check=True)
    return oracle.load_library(str(so))


def _rand(shape, seed):
    return torch.randn(shape, generator=torch.Generator().manual_seed(seed), dtype=torch.float32)


def _battery(lib) -> bool:
    """True when the build passes every quick pin."""
    att = lambda *a, **kw: oracle.attention(*a, lib=lib, **kw)  # noqa: E731
    # closed forms
    with open(os.path.join(HERE, "golden", "closed_forms.json")) as f:
        for gc in json.load(f)["cases"]:
            out = att(np.array(gc["q"], np.float32), np.array(gc["k"], np.float32),
                      np.array(gc["v"], np.float32), pos_offset=gc["pos_offset"],
                      mask_mode=gc["mask_mode"], window=gc["window"], key_lens=gc["key_lens"],
                      scale=gc["scale"])
            if np.max(np.abs(out - np.array(gc["expected"]))) > gc["tol"]:
                return False
    # library routine: GQA + key padding, and causal with an offset
    q, k, v = _rand((2, 4, 9, 8), 1), _rand((2, 2, 12, 8), 2), _rand((2, 2, 12, 8), 3)
    lens = torch.tensor([12, 7])
    mask = (torch.arange(12)[None, :] < lens[:, None])[:, None, None, :]
    ref = F.scaled_dot_product_attention(q.double(), k.double().repeat_interleave(2, 1),
                                         v.double().repeat_interleave(2, 1), attn_mask=mask, scale=0.3)
    if np.max(np.abs(att(q, k, v, key_lens=lens.int(), scale=0.3) - ref.numpy())) > 1e-10:
        return False
    cm = torch.ones(9, 12, dtype=torch.bool).tril(diagonal=3)
    ref = F.scaled_dot_product_attention(q.double(), k.double().repeat_interleave(2, 1),
                                         v.double().repeat_interleave(2, 1), attn_mask=cm, scale=0.3)
    if np.max(np.abs(att(q, k, v, mask_mode=1, pos_offset=3, scale=0.3) - ref.numpy())) > 1e-10:
        return False
    # visible sets of the windowed modes (scale 0 + one-hot V)
    eye = np.eye(12, dtype=np.float32)[None, None]
    z = np.zeros((1, 1, 6, 12), np.float32)
    for mode, w, rule in ((2, 4, lambda p, j: abs(p - j) <= 2), (2, 5, lambda p, j: abs(p - j) <= 2),
                         (3, 4, lambda p, j: p - 4 < j <= p)):
        out = att(z, eye, eye, mask_mode=mode, window=w, pos_offset=2, scale=0.0)[0, 0]
        for i in range(6):
            vis = [j for j in range(12) if rule(2 + i, j)]
            exp = np.zeros(12)
            exp[vis] = 1.0 / len(vis)
            if np.max(np.abs(out[i] - exp)) > 1e-15:
                return False
    return True


def test_unmodified_source_passes_battery(tmp_path):
    assert _battery(_build(tmp_path, open(SRC).read(), "orig"))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found once"
    assert not _battery(_build(tmp_path, text.replace(old, new), name))
