"""The FP32 / SFU rate kernels (gsr_peak_kernel) that give the raster kernels'
roofline its denominators: the lane-operation count they report, rates within
reach of the formula SMs x lanes x clock, and their argument checks."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsr_ctx():
    import gaussian_splatting_tile_bin_gb300 as gsr
    ctx = gsr.Context(0)
    yield gsr, ctx
    ctx.close()


def _rate(gsr, ctx, kind, iters, sink):
    stream = torch.cuda.current_stream()
    for _ in range(2):
        gsr.peak_kernel(ctx, kind, iters, sink)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    ops = gsr.peak_kernel(ctx, kind, iters, sink)
    b.record(stream)
    b.synchronize()
    return ops, ops / (a.elapsed_time(b) * 1e-3)


# Lanes per SM per clock: 128 FP32 lanes; the SFU runs ex2 at 32 lanes per
# clock on GB300 (measured: an earlier expectation of 16 failed this test at
# twice that rate).
@pytest.mark.parametrize("kind,lanes,iters", [("ffma", 128, 16384), ("ex2", 32, 2048)])
def test_rate_is_near_the_formula(gsr_ctx, kind, lanes, iters):
    gsr, ctx = gsr_ctx
    sink = torch.zeros(1, dtype=torch.float32, device="cuda:0")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ops, rate = _rate(gsr, ctx, kind, iters, sink)
    # 8 CTAs of 256 threads per SM, 16 chains per round, rounds a multiple of 8
    assert ops == sms * 8 * 256 * iters * 16
    formula_at_max = sms * lanes * 2070e6
    # below the formula at the part's maximum clock (plus timing slack), and
    # not far below it: the kernel keeps the pipe busy
    assert 0.6 * formula_at_max < rate < 1.1 * formula_at_max, (kind, rate / formula_at_max)
    assert float(sink.item()) == 0.0


def test_bad_arguments_are_rejected(gsr_ctx):
    gsr, ctx = gsr_ctx
    sink = torch.zeros(1, dtype=torch.float32, device="cuda:0")
    with pytest.raises(gsr.GsrError):
        gsr.peak_kernel(ctx, "ffma", 0, sink)
    with pytest.raises(gsr.GsrError):
        gsr.peak_kernel(ctx, "ex2", (1 << 24) + 1, sink)
    from gaussian_splatting_tile_bin_gb300 import _abi
    import ctypes
    ops = ctypes.c_uint64()
    rc = _abi.lib.gsr_peak_kernel(ctx._h, 7, 8, ctypes.c_void_p(sink.data_ptr()), ctypes.byref(ops), None)
    assert rc == _abi.GSR_ERR_INVALID_ARG
