"""tcgen05/TMA building blocks: one 128x128x128 bf16 tile product per operand
layout, compared with torch.matmul (fp32 accumulate) on the GPU."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jfa():
    import bwd_jagged_flashattention_gb300 as jfa
    return jfa


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
def test_tile_mma(jfa, mode):
    g = torch.Generator().manual_seed(mode)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    c, status = jfa.selftest_mma(mode, a, b)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    af, bf = a.float(), b.float()
    ref = {0: af @ bf.T, 1: af @ bf, 2: af @ bf, 3: af.T @ bf, 4: af @ bf}[mode]
    err = (c - ref).abs().max().item()
    assert err <= 1e-2 * ref.abs().max().item(), f"mode {mode}: max err {err}"
