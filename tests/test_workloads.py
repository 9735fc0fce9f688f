"""The seeded synthetic workloads: determinism and the shape facts they stand in for."""
import numpy as np
import pytest

import gen
import oracle


@pytest.mark.parametrize("name", ["tiny", "small", "lego_early"])
def test_deterministic_and_well_formed(name):
    a, b = gen.make(name), gen.make(name)
    assert np.array_equal(a.splats, b.splats) and np.array_equal(a.dl_dout, b.dl_dout)
    s = a.splats
    assert s.dtype == np.float32 and s.shape[1] == 9
    assert np.all(np.isfinite(s)) and np.all(a.depths > 0)
    det = s[:, 2].astype(np.float64) * s[:, 4] - s[:, 3].astype(np.float64) ** 2
    assert np.all(s[:, 2] > 0) and np.all(det > 0)
    assert np.all((s[:, 8] > 0) & (s[:, 8] < 1))
    assert np.all((s[:, 5:8] >= 0) & (s[:, 5:8] <= 1))
    assert np.all(a.dl_dout[:, 3] == 0)
    assert a.dl_dout.shape == (a.width * a.height, 4)


def test_config_sizes():
    sizes = {"tiny": (64, 64, 256), "small": (256, 256, 10_000),
             "lego_early": (800, 800, 83_734), "lego_final": (800, 800, 409_660)}
    for name, (w, h, n) in sizes.items():
        wl = gen.make(name)
        assert (wl.width, wl.height, wl.n) == (w, h, n)


def test_small_low_opacity_subset():
    s = gen.small().splats
    assert abs(np.mean(s[:, 8] < 0.01) - 0.15) < 0.01


def test_lego_final_shape():
    """~94% of splat-pixel evaluations contribute nothing ("p2-w1-warp-sparse-skip",
    body) and the tile-pair count stays within 16 N."""
    wl = gen.lego_final()
    keys, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    assert len(keys) <= 16 * wl.n
    c = oracle.forward(wl.splats, idx, ranges, wl.width, wl.height)["counters"]
    frac = 1.0 - c["n_contrib"] / c["n_eval"]
    assert 0.90 <= frac <= 0.97, frac


def test_lego_far_crowds_a_few_tiles():
    """lego_final from four times the distance: the same splats, footprints a
    quarter the size, depth order kept.  Its heaviest tile carries more than ten
    times a balanced share of 608 CTA slots (152 SMs x 4) of the per-pixel work
    (the sum of last_contributor over the tile), the case a split of long
    lists is for."""
    near, far = gen.lego_final(), gen.lego_far()
    assert far.n == near.n
    assert np.array_equal(np.argsort(far.depths, kind="stable"), np.argsort(near.depths, kind="stable"))
    s = far.splats.astype(np.float64)
    assert np.all(np.isfinite(s)) and np.all(s[:, 2] * s[:, 4] - s[:, 3] ** 2 > 0)
    keys, idx, ranges = oracle.bin_splats(far.splats, far.depths, far.width, far.height)
    last = oracle.forward(far.splats, idx, ranges, far.width, far.height)["last"].astype(np.int64)
    cost = last.reshape(50, 16, 50, 16).transpose(0, 2, 1, 3).reshape(2500, 256).sum(axis=1)
    share = cost.sum() / 608.0
    assert cost.max() > 10.0 * share
    assert len(keys) < len(oracle.bin_splats(near.splats, near.depths, 800, 800)[0])


def test_lego_pages_matches_the_pages_pair_density():
    """lego_final's splats with smaller footprints: about 2.4 pairs per splat,
    the density of the pages' final checkpoint (969,838 pairs for 407,267
    splats, "forward/adam audit" section 3, staging read)."""
    wl = gen.make("lego_pages")
    assert (wl.width, wl.height, wl.n) == (800, 800, 409_660)
    keys, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    assert 2.3 <= len(keys) / wl.n <= 2.5
    assert abs(len(keys) / wl.n - 969_838 / 407_267) < 0.05
