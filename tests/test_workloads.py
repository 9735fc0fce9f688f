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
