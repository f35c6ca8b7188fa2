"""The two 2^x routines the softmax uses, against exact 2^x of the same float inputs."""
import pytest
import torch

import head_attention_attn_gb300 as attn

pytestmark = pytest.mark.gpu


def test_exp2_routines_meet_their_error_bounds():
    from head_attention_attn_gb300 import build
    build.build_library()
    x = torch.linspace(-125.0, 64.0, 3_000_001, dtype=torch.float32)
    x = torch.cat([x, torch.tensor([0.0, 0.5, -0.5, 1.0, -1.0, 8.0, -124.5, 63.9])])
    yp, yu = attn.selftest_exp2(x.cuda())
    torch.cuda.synchronize()
    exact = torch.exp2(x.double())
    rel_poly = ((yp.double().cpu() - exact) / exact).abs().max().item()
    rel_unit = ((yu.double().cpu() - exact) / exact).abs().max().item()
    assert rel_poly < 1e-4, rel_poly
    assert rel_unit < 1e-6, rel_unit
    # below the clamp the polynomial returns 2^-125 (within its error bound) and the unit flushes to zero
    ninf = torch.tensor([-float("inf"), -200.0], device="cuda")
    yp, yu = attn.selftest_exp2(ninf)
    assert torch.all((yp.double() / 2.0 ** -125 - 1).abs() < 1e-4) and torch.all(yu == 0)
