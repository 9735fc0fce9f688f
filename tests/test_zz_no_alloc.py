"""The backward entry point that allocates nothing.

Some callers cannot call cudaMalloc: their device memory is reserved up front
by another allocator, or they run a loop that must not stall or fail halfway
(cudaMalloc may synchronise the device).  gsr_rasterize_backward_noalloc serves
them with a fixed device array as its accumulator.  This test calls it through
the C ABI, twice in a row with different splat counts, and checks each result
against gsr_rasterize_backward within the gradient tolerance of the other GPU
tests, and the first (the small set) against the CPU oracle as well.  It also
checks that a splat count above the array's limit is refused.

This file is named to be collected last, and it builds everything it needs, so
it runs the same alone in a fresh process as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
from gpu_helpers import GRAD_ATOL, GRAD_RTOL, as_result, check_backward, run_oracle, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


def _noalloc_fn(gsr):
    from gaussian_splatting_tile_bin_gb300 import _abi
    fn = _abi.lib.gsr_rasterize_backward_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [P, P, ctypes.c_int32, ctypes.POINTER(_abi._Bins), P, P, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def _prepare(gsr, ctx, wl):
    sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
    bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
    out, final_t, last = gsr.rasterize_forward(ctx, sp, bins)
    return sp, dl, bins, out, final_t, last


def _call_noalloc(fn, ctx, sp, bins, dl, final_t, last, grad):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctx._h, ctypes.c_void_p(sp.data_ptr()), sp.shape[0], ctypes.byref(bins.raw),
              ctypes.c_void_p(dl.data_ptr()), ctypes.c_void_p(final_t.data_ptr()),
              ctypes.c_void_p(last.data_ptr()), ctypes.c_void_p(grad.data_ptr()), stream)


def test_noalloc_backward_matches_backward_on_two_calls(gsr):
    fn = _noalloc_fn(gsr)
    ctx = gsr.Context(0)
    try:
        # Two calls in a row; the second is larger, so it must clear and reuse
        # more of the shared array than the first left behind.
        for wl in (gen.small(), gen.lego_early()):
            sp, dl, bins, out, final_t, last = _prepare(gsr, ctx, wl)
            ref = gsr.rasterize_backward(ctx, sp, bins, dl, final_t, last).cpu().numpy()
            grad = torch.full((wl.n, 9), float("nan"), dtype=torch.float32, device="cuda:0")
            rc = _call_noalloc(fn, ctx, sp, bins, dl, final_t, last, grad)
            assert rc == 0, gsr._abi.lib.gsr_last_error(ctx._h)
            got = grad.cpu().numpy()
            assert np.all(np.isfinite(got))
            assert np.all(np.abs(got - ref) <= GRAD_ATOL + GRAD_RTOL * np.abs(ref)), wl.name
            if wl.name == "small":
                check_backward(as_result(out, final_t, last, got), run_oracle(wl))
    finally:
        ctx.close()


def test_noalloc_backward_refuses_too_many_splats(gsr):
    from gaussian_splatting_tile_bin_gb300 import _abi
    fn = _noalloc_fn(gsr)
    ctx = gsr.Context(0)
    try:
        wl = gen.lego_final()   # 409,660 splats: above the fixed array's 131,072
        sp, dl, bins, out, final_t, last = _prepare(gsr, ctx, wl)
        grad = torch.zeros((wl.n, 9), dtype=torch.float32, device="cuda:0")
        rc = _call_noalloc(fn, ctx, sp, bins, dl, final_t, last, grad)
        assert rc == 1
        assert b"GSR_NOALLOC_MAX_SPLATS" in _abi.lib.gsr_last_error(ctx._h)
    finally:
        ctx.close()
