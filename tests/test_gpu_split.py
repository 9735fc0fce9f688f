"""The split of crowded tiles (GSR_OPT_SPLIT, on by default, and
GSR_OPT_SPLIT_FORWARD, off by default).

Forward: a list longer than a head of max(1024, half the pairs per CTA slot)
positions stops there; the rest of an unfinished tile runs as 512-position chunks
composited from transmittance 1, each pixel's stop is found from the chunk
products and replayed from the true transmittance, and the tile's last replay
assembles it.  Backward: the forward records each pixel's transmittance and
the colour behind every 512th position of a tile's list, and the backward that
follows it runs long lists as segments of a multiple of 512 positions (sized on
the device from the frame's work), each its own CTA starting from those states.

Parity with the oracle on the crowded-tile sets (lego_final seen from 4 and 8
times the distance: a few dozen tiles with lists of tens of thousands of
splats), on a small fixture whose pixels stop inside the head, inside the
chunks and not at all, over a ragged image; the backward split alone leaves
the forward's transmittance and last_contrib bits unchanged; the forward split
moves them only by rounding, and nothing on a frame without crowded tiles;
repeated forwards give the same bits; the backward falls back to one CTA per
tile when it is not given the buffers of the forward that recorded the states.
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
    for det, fwd in ((False, False), (True, False), (False, True), (True, True)):
        ctx.set_option("deterministic", det)
        ctx.set_option("split_forward", fwd)
        g = run_gpu(gsr, ctx, wl)
        check_bins(g, o)
        fs = check_forward(g, o)
        bs = check_backward(g, o)
        record_stats(f"lego_far x{distance:g}{' det' if det else ''}{' split fwd' if fwd else ''}",
                     forward=fs, backward=bs)
    ctx.set_option("deterministic", False)
    ctx.set_option("split_forward", False)


def crowded_fixture(seed=11, n=6000, width=40, height=20):
    """Six tiles (a ragged 40 x 20 image) with lists of 4,000-6,000 wide,
    faint splats whose opacity grows to the right: pixels on the right stop
    within the forward's 1,024-position head, those in the middle inside its
    chunks, and a quarter on the left never."""
    rng = np.random.default_rng(seed)
    sp = np.zeros((n, 9), np.float32)
    sp[:, 0] = rng.uniform(-4, 40, n)
    sp[:, 1] = rng.uniform(-2, 20, n)
    std = rng.uniform(3, 12, n)
    sp[:, 2] = sp[:, 4] = 1.0 / std ** 2
    sp[:, 3] = rng.uniform(-0.3, 0.3, n) / std ** 2
    sp[:, 5:8] = rng.uniform(0, 1, (n, 3))
    sp[:, 8] = np.clip(0.0012 * np.exp(rng.uniform(0, 1.5, n)) * (1 + np.maximum(sp[:, 0] - 16, 0) / 0.8), 0, 0.9)
    return gen.from_arrays("crowded", width, height, sp, rng.uniform(1, 9, n).astype(np.float32), seed=seed)


def test_forward_split_fixture_parity(gsr, ctx):
    wl = crowded_fixture()
    o = run_oracle(wl)
    T, last = o["fwd"]["final_T"], o["fwd"]["last"]
    stopped = T < 3e-4
    assert np.any(stopped & (last < 1024)) and np.any(stopped & (last > 1024)) and np.any(~stopped)
    ctx.set_option("split_forward", True)
    try:
        for det in (False, True):
            ctx.set_option("deterministic", det)
            g = run_gpu(gsr, ctx, wl)
            check_bins(g, o)
            fs = check_forward(g, o)
            bs = check_backward(g, o)
            record_stats(f"crowded fixture{' det' if det else ''}", forward=fs, backward=bs)
    finally:
        ctx.set_option("deterministic", False)
        ctx.set_option("split_forward", False)


def _runs(gsr, ctx, wl, settings):
    runs = {}
    for name, (split, fwd) in settings.items():
        ctx.set_option("split", split)
        ctx.set_option("split_forward", fwd)
        runs[name] = run_gpu(gsr, ctx, wl)
    ctx.set_option("split", True)
    ctx.set_option("split_forward", False)
    return runs


def _same_bits(a, b, keys):
    for k in keys:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


def _grads_close(a, b):
    a, b = a["grad"].astype(np.float64), b["grad"].astype(np.float64)
    assert np.all(np.abs(a - b) <= 1e-4 + 1e-4 * np.abs(b))


@pytest.mark.parametrize("name", ["lego_far", "stress"])
def test_backward_split_keeps_the_forward_bits(gsr, ctx, name):
    wl = gen.make(name)
    runs = _runs(gsr, ctx, wl, {"off": (False, False), "bwd": (True, False)})
    # T and last_contrib are the same bits; a long list's colour is summed per
    # segment (the segments' colours are what the backward starts from), so it
    # differs from the running sum by float rounding only
    _same_bits(runs["bwd"], runs["off"], ("final_T", "last"))
    assert np.abs(runs["bwd"]["out"] - runs["off"]["out"]).max() <= 2e-6
    _grads_close(runs["bwd"], runs["off"])


def test_forward_split_moves_results_by_rounding_only(gsr, ctx):
    wl = gen.lego_far()
    runs = _runs(gsr, ctx, wl, {"bwd": (True, False), "both": (True, True)})
    a, b = runs["both"], runs["bwd"]
    # the split ran: the transmittance past the heads rounds as chunk products
    assert np.any(a["final_T"] != b["final_T"])
    # a stop moves only where next_T lies within rounding of the threshold
    # (the parity tests check each such pixel against the oracle's forced
    # replay); elsewhere colour and transmittance move by rounding
    same = a["last"] == b["last"]
    assert np.mean(~same) < 1e-3
    assert np.abs(a["final_T"] - b["final_T"])[same].max() <= 1e-5
    assert np.abs(a["out"] - b["out"])[same].max() <= 1e-5
    # a frame whose lists are all shorter than the head does not split
    # (stress: head 15,872 positions, longest list 14,478)
    wl = gen.stress()
    runs = _runs(gsr, ctx, wl, {"bwd": (True, False), "both": (True, True)})
    _same_bits(runs["both"], runs["bwd"], ("out", "final_T", "last", "grad"))


def test_repeated_forwards_give_the_same_bits(gsr, ctx):
    """The chunk queue is cleared by each forward's last replay CTA: forwards
    of split and unsplit frames in any order give the same bits."""
    far, early = gen.lego_far(), gen.lego_early()
    ctx.set_option("deterministic", True)
    ctx.set_option("split_forward", True)
    try:
        first = run_gpu(gsr, ctx, far)
        run_gpu(gsr, ctx, early, backward=False)
        again = run_gpu(gsr, ctx, far)
        again2 = run_gpu(gsr, ctx, far)
    finally:
        ctx.set_option("deterministic", False)
        ctx.set_option("split_forward", False)
    for r in (again, again2):
        _same_bits(r, first, ("out", "final_T", "last", "grad"))


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
