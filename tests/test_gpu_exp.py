"""The raster kernels' exponential against float64 exp, through gsr_exp_neg.

alpha = min(0.999, color_a exp(-sigma)) is evaluated for 0 <= sigma < 5.55
only ("W1 warp sparse skip + exp-skip", section 1: larger sigma is skipped).
The kernels' exp(-s) must stay within 3 ulp of the correctly rounded value
over that whole range: the forward's 1e-5 budget and the oracle's 6e-7
relative knife-edge margin for alpha both rest on it.  A dense sample of every
float in [0, 5.55] (a fixed stride through their bit patterns, plus both ends)
is compared with torch's float64 exp rounded to float.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


def test_exp_neg_within_3_ulp_over_the_sigma_range(gsr):
    from gaussian_splatting_tile_bin_gb300 import _abi
    top = int(np.float32(5.55).view(np.int32))
    bits = torch.arange(0, top + 1, 61, dtype=torch.int32, device="cuda:0")
    bits = torch.cat([bits, torch.tensor([1, 2, top - 1, top], dtype=torch.int32, device="cuda:0")])
    s = bits.view(torch.float32)
    ctx = gsr.Context(0)
    try:
        out = _abi.exp_neg(ctx, s)
        torch.cuda.synchronize()
    finally:
        ctx.close()
    ref = torch.exp(-s.double())
    ulps = (out.view(torch.int32).long() - ref.float().view(torch.int32).long()).abs()
    rel = ((out.double() - ref).abs() / ref).max().item()
    assert out[0].item() == 1.0  # exp(-0)
    assert int(ulps.max().item()) <= 3, int(ulps.max().item())
    assert rel < 2.5e-7, rel


def test_exp_neg_rejects_bad_arguments(gsr):
    from gaussian_splatting_tile_bin_gb300 import _abi
    ctx = gsr.Context(0)
    try:
        rc = _abi.lib.gsr_exp_neg(ctx._h, None, None, -1, None)
        assert rc == _abi.GSR_ERR_INVALID_ARG
    finally:
        ctx.close()
