"""The split backward of long tile lists (GSR_OPT_SPLIT).

The forward records each pixel's transmittance and the colour behind every
512th position of a tile's list; the backward that follows it runs long lists
as segments of a multiple of 512 positions (sized on the device from the
frame's work), each its own CTA starting from those states.
Parity with the oracle on the crowded-tile sets (lego_final seen from 4 and 8
times the distance: a few dozen tiles with lists of tens of thousands of
splats) and on the stress set; the forward's transmittance and last_contrib
are the same bits with the split on or off; the backward falls back to one
CTA per tile when it is not given the buffers of the forward that recorded the
states.
"""
import numpy as np
import pytest
import torch

import gen
from gpu_helpers import (as_result, check_backward, check_bins, check_forward, record_stats, run_gpu, run_oracle,
                         to_dev)

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


@pytest.mark.parametrize("distance", [4.0, 8.0])
def test_crowded_tiles_parity(gsr, ctx, distance):
    wl = gen.lego_far(distance=distance)
    o = run_oracle(wl)
    assert int(np.max(o["ranges"][:, 1] - o["ranges"][:, 0])) > 8 * 512      # lists that split
    for det in (False, True):
        ctx.set_option("deterministic", det)
        g = run_gpu(gsr, ctx, wl)
        check_bins(g, o)
        fs = check_forward(g, o)
        bs = check_backward(g, o)
        record_stats(f"lego_far x{distance:g}{' det' if det else ''}", forward=fs, backward=bs)
    ctx.set_option("deterministic", False)


@pytest.mark.parametrize("name", ["lego_far", "stress"])
def test_split_on_and_off_agree(gsr, ctx, name):
    wl = gen.make(name)
    runs = {}
    for on in (True, False):
        ctx.set_option("split", on)
        runs[on] = run_gpu(gsr, ctx, wl)
    ctx.set_option("split", True)
    # T and last_contrib are the same bits; a long list's colour is summed per
    # segment (the segments' colours are what the backward starts from), so it
    # differs from the running sum by float rounding only
    for k in ("final_T", "last"):
        assert np.array_equal(runs[True][k].view(np.uint8), runs[False][k].view(np.uint8)), k
    assert np.abs(runs[True]["out"] - runs[False]["out"]).max() <= 2e-6
    a, b = runs[True]["grad"].astype(np.float64), runs[False]["grad"].astype(np.float64)
    assert np.all(np.abs(a - b) <= 1e-4 + 1e-4 * np.abs(b))


def test_backward_without_the_forward_states_falls_back(gsr, ctx):
    """The backward splits only over the forward buffers that recorded the
    states; given copies (or after another binning) it runs one CTA per tile,
    with the same results within float rounding."""
    wl = gen.lego_far()
    sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
    bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
    out, fT, last = gsr.rasterize_forward(ctx, sp, bins)
    split = gsr.rasterize_backward(ctx, sp, bins, dl, fT, last).cpu().numpy()
    fT2, last2 = fT.clone(), last.clone()
    launches = ctx.launch_count()
    copied = gsr.rasterize_backward(ctx, sp, bins, dl, fT2, last2).cpu().numpy()
    # tile cost, tile order, backward, conversion: no plan kernel
    assert ctx.launch_count() - launches == 4
    assert np.all(np.abs(split.astype(np.float64) - copied) <= 1e-4 + 1e-4 * np.abs(copied))
    o = run_oracle(wl)
    check_backward(as_result(out, fT2, last2, copied), o)
