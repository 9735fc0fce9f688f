"""Failure detection through the C ABI, with the failure made on the host.

An allocation failure is injected with the context's test hook (the next
device allocation fails as if the GPU were out of memory).  The call must
report GSR_ERR_OOM with a message, leave the context usable, and the next
call must allocate and give the oracle's results.  No GPU fault is involved.
"""
import numpy as np
import pytest
import torch

import gen
from gpu_helpers import as_result, check_backward, check_bins, check_forward, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

GSR_ERR_OOM = 3


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


def test_binning_reports_an_allocation_failure_and_recovers(gsr):
    wl = gen.small()
    sp, dp = to_dev(wl.splats), to_dev(wl.depths)
    ctx = gsr.Context(0)
    try:
        ctx.set_option("fail_next_alloc", 1)
        with pytest.raises(gsr.GsrError) as err:
            gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        assert err.value.code == GSR_ERR_OOM and "cudaMalloc failed" in str(err.value)
        g = run_gpu(gsr, ctx, wl)
        o = run_oracle(wl)
        check_bins(g, o)
        check_forward(g, o)
        check_backward(g, o)
    finally:
        ctx.close()


def test_arena_growth_reports_an_allocation_failure_and_recovers(gsr):
    small, large = gen.tiny(), gen.lego_early()
    ctx = gsr.Context(0)
    try:
        run_gpu(gsr, ctx, small)                      # arena sized for the tiny set
        ctx.set_option("fail_next_alloc", 1)          # the growth for the large set fails
        sp, dp = to_dev(large.splats), to_dev(large.depths)
        with pytest.raises(gsr.GsrError) as err:
            gsr.bin_splats(ctx, sp, dp, large.width, large.height)
        assert err.value.code == GSR_ERR_OOM
        g = run_gpu(gsr, ctx, large)
        o = run_oracle(large, backward=False)
        check_bins(g, o)
        check_forward(g, o)
    finally:
        ctx.close()


def test_backward_reports_an_allocation_failure_and_recovers(gsr):
    wl = gen.small()
    sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
    ctx = gsr.Context(0)
    try:
        bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        out, final_t, last = gsr.rasterize_forward(ctx, sp, bins)
        ctx.set_option("fail_next_alloc", 1)          # the gradient accumulator
        with pytest.raises(gsr.GsrError) as err:
            gsr.rasterize_backward(ctx, sp, bins, dl, final_t, last)
        assert err.value.code == GSR_ERR_OOM
        grad = gsr.rasterize_backward(ctx, sp, bins, dl, final_t, last).cpu().numpy()
        o = run_oracle(wl)
        check_backward(as_result(out, final_t, last, grad), o)
        assert np.all(np.isfinite(grad))
    finally:
        ctx.close()


def test_deterministic_backward_reports_an_allocation_failure_and_recovers(gsr):
    """The deterministic mode allocates its exponent table on first use: a
    failure there is reported and the next call recovers."""
    wl = gen.small()
    sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
    ctx = gsr.Context(0)
    try:
        bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        out, final_t, last = gsr.rasterize_forward(ctx, sp, bins)
        gsr.rasterize_backward(ctx, sp, bins, dl, final_t, last)   # accumulator and tile order allocated
        ctx.set_option("deterministic", True)
        ctx.set_option("fail_next_alloc", 1)                       # the exponent table
        with pytest.raises(gsr.GsrError) as err:
            gsr.rasterize_backward(ctx, sp, bins, dl, final_t, last)
        assert err.value.code == GSR_ERR_OOM and "deterministic" in str(err.value)
        grad = gsr.rasterize_backward(ctx, sp, bins, dl, final_t, last).cpu().numpy()
        check_backward(as_result(out, final_t, last, grad), run_oracle(wl))
    finally:
        ctx.close()
