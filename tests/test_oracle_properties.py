"""Property-based pins of the oracle (hypothesis; skipped where it is not
installed): on arbitrary small inputs the binning equals the numpy route
(emission in plain loops, numpy's lexsort, searchsorted ranges), and the tiled
forward equals the untiled brute force bit for bit."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from test_oracle_pins import _numpy_binning  # noqa: E402


@st.composite
def splat_sets(draw):
    w = draw(st.integers(1, 80))
    h = draw(st.integers(1, 80))
    n = draw(st.integers(0, 60))
    seed = draw(st.integers(0, 2**32 - 1))
    rng = np.random.Generator(np.random.PCG64(seed))
    s = np.zeros((n, 9), dtype=np.float32)
    s[:, 0] = rng.uniform(-20, w + 20, n)
    s[:, 1] = rng.uniform(-20, h + 20, n)
    std1 = np.exp(rng.uniform(np.log(0.3), np.log(30.0), n))
    std2 = std1 / np.exp(rng.uniform(0.0, np.log(20.0), n))
    th = rng.uniform(0, np.pi, n)
    ct, sn = np.cos(th), np.sin(th)
    sxx = ct * ct * std1 ** 2 + sn * sn * std2 ** 2
    syy = sn * sn * std1 ** 2 + ct * ct * std2 ** 2
    sxy = ct * sn * (std1 ** 2 - std2 ** 2)
    det = sxx * syy - sxy * sxy
    s[:, 2], s[:, 3], s[:, 4] = syy / det, -sxy / det, sxx / det
    s[:, 5:8] = rng.uniform(0, 1, (n, 3))
    s[:, 8] = rng.uniform(0, 1, n)
    levels = draw(st.sampled_from([None, 3]))
    d = (rng.integers(1, 4, n) if levels else rng.uniform(0.5, 20.0, n)).astype(np.float32)
    return s, d, w, h


@settings(max_examples=60, deadline=None)
@given(splat_sets())
def test_binning_equals_numpy_route(case):
    s, d, w, h = case
    k, i, r = oracle.bin_splats(s, d, w, h)
    k2, i2, r2 = _numpy_binning(s, d, w, h)
    assert np.array_equal(k, k2) and np.array_equal(i, i2) and np.array_equal(r, r2)


@settings(max_examples=40, deadline=None)
@given(splat_sets())
def test_tiled_forward_equals_untiled(case):
    s, d, w, h = case
    _, i, r = oracle.bin_splats(s, d, w, h)
    a = oracle.forward(s, i, r, w, h)
    b = oracle.forward_untiled(s, d, w, h)
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["final_T"], b["final_T"])
    assert np.array_equal(a["last"], b["last"])
