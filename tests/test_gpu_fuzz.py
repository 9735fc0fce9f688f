"""Randomised cases (gen.random_case: odd image sizes, splats off the image,
thin and huge splats, exact depth ties, culled values, empty inputs) through
the whole CUDA path against the oracle, in the default and the deterministic
backward.

Every difference beyond tolerance must be reproduced by the oracle with
decisions within their rounding uncertainty taken the other way (a forced
replay).  Dense random overlap makes such decisions more common than on the
configs: one pixel whose stop decision (T against 1e-4) flips changes the
terms of every splat behind it there, and the forced replay carries that
flip into every one of those splats' gradients."""
import numpy as np
import pytest
import torch

import gen
from gpu_helpers import check_backward, check_bins, check_forward, record_stats, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


@pytest.fixture(scope="module")
def ctx(gsr):
    c = gsr.Context(0)
    yield c
    c.close()


@pytest.mark.parametrize("seed", range(24))
def test_random_case(gsr, ctx, seed):
    wl = gen.random_case(seed)
    o = run_oracle(wl)
    for det in (False, True):
        ctx.set_option("deterministic", det)
        g = run_gpu(gsr, ctx, wl)
        check_bins(g, o)
        fs = check_forward(g, o)
        bs = check_backward(g, o)
        record_stats(f"random{seed}{' det' if det else ''}", forward=fs, backward=bs)
    ctx.set_option("deterministic", False)
