"""The parity checker's knife-edge rule, on the CPU.

A result that differs from the oracle passes only when a forced replay of the
oracle, with decisions that lie within their rounding uncertainty taken the
other way, reproduces it.  Here the "GPU" results are the oracle's own forced
replays (what a correct implementation that rounds differently may produce),
and a planted error of 1e-3 on top of them must fail, on a flagged pixel and a
flagged splat alike.
"""
import numpy as np
import pytest

import gen
import oracle
from gpu_helpers import EPS_ALPHA, FWD_TOL, check_backward, check_forward, run_oracle


def _fake(o, flips):
    """What an implementation that took the decisions `flips` names the other
    way computes: the oracle's forced forward and backward."""
    wl = o["wl"]
    f = oracle.forward_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, flips,
                              eps_alpha=EPS_ALPHA)
    b = oracle.backward_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, wl.dl_dout, flips,
                               eps_alpha=EPS_ALPHA)
    assert f["refused"] == 0 and b["refused"] == 0
    return {"out": f["out"], "final_T": f["final_T"], "last": f["last"], "grad": b["grad"].astype(np.float32)}


def _visible_flip(o):
    """A decision within its uncertainty whose flip moves its pixel beyond the
    forward tolerance or changes its last_contrib."""
    wl, f = o["wl"], o["fwd"]
    for p in np.nonzero(f["margin"] < 1.0)[0]:
        px, py = p % wl.width, p // wl.width
        base, last, dec, _ = oracle.pixel_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, px, py,
                                                 None, eps_alpha=EPS_ALPHA)
        for d in dec:
            t = oracle.flip_table([(p, d["pos"], d["type"])])
            o5, l2, _, refused = oracle.pixel_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, px,
                                                     py, t, eps_alpha=EPS_ALPHA)
            if refused == 0 and (np.abs(o5 - base).max() > FWD_TOL or l2 != last):
                return int(p), t
    raise AssertionError("no visible knife-edge in this workload")


@pytest.fixture(scope="module")
def small_case():
    o = run_oracle(gen.small())
    p, flips = _visible_flip(o)
    return o, p, flips


def test_a_flipped_decision_is_explained(small_case):
    o, p, flips = small_case
    g = _fake(o, flips)
    fs = check_forward(g, o)
    assert fs["flipped_px"] >= 1 and fs["max_abs"] <= FWD_TOL
    bs = check_backward(g, o)
    assert bs["flips"] >= 1


def test_a_planted_error_on_a_flagged_pixel_fails(small_case):
    o, p, flips = small_case
    g = _fake(o, flips)
    g["out"] = g["out"].copy()
    g["out"][p, 1] += 1e-3                 # the flipped pixel itself
    with pytest.raises(AssertionError):
        check_forward(g, o)
    g = _fake(o, flips)
    other = [q for q in np.nonzero(o["fwd"]["margin"] < 1.0)[0] if q != p][0]
    g["final_T"] = g["final_T"].copy()
    g["final_T"][other] += 1e-3            # a flagged pixel that did not flip
    with pytest.raises(AssertionError):
        check_forward(g, o)


def test_a_planted_error_on_a_flagged_splat_fails(small_case):
    o, p, flips = small_case
    g = _fake(o, flips)
    s = int(np.nonzero(o["bwd"]["knife"])[0][0])
    g["grad"] = g["grad"].copy()
    g["grad"][s, 8] += np.float32(1e-3) + np.float32(1e-4) * abs(g["grad"][s, 8])
    with pytest.raises(AssertionError):
        check_backward(g, o)


def _hidden_fixture(kind):
    """Splats on a 16x16 image, all hit at pixel (8, 8); the splat under test
    sits exactly at that pixel, so sigma = 0 and raw = color_a there.
      alpha: three splats of alpha 0.9 in front leave T = 1e-3, then the splat
             under test with color_a = 1/255 (alpha exactly at the cut: its
             colour is 4e-6 of the pixel, below the forward tolerance), then a
             splat of alpha 0.5 behind it;
      clamp: the splat under test with color_a = 0.999 (raw exactly at the
             clamp: alpha is 0.999 either way), then a splat of alpha 0.5.
    Returns the workload and the tested splat's position (= index)."""
    conic = [0.02, 0.0, 0.02]
    behind = [7.0, 9.0, *conic, 0.4, 0.8, 0.6, 0.5]
    if kind == "alpha":
        rows = [[8.0, 8.0, *conic, 0.3 * k, 0.5, 0.9, 0.9] for k in range(3)]
        rows += [[8.0, 8.0, *conic, 0.2, 0.5, 0.9, np.float32(1.0) / np.float32(255.0)], behind]
        tested = 3
    else:
        rows = [[8.0, 8.0, *conic, 0.7, 0.1, 0.3, 0.999], behind]
        tested = 0
    splats = np.array(rows, dtype=np.float32)
    depths = np.arange(1, len(rows) + 1, dtype=np.float32)
    return gen.from_arrays(f"hidden_{kind}", 16, 16, splats, depths, seed=3), tested


@pytest.mark.parametrize("kind,typ", [("alpha", oracle.DEC_ALPHA), ("clamp", oracle.DEC_CLAMP)])
def test_a_hidden_flip_is_found(kind, typ):
    """A decision at the cut or the clamp that leaves the pixel's colour
    within tolerance and its last_contrib unchanged still moves the splat's
    own gradient; the checker finds that flip, and a planted error on top of
    it still fails."""
    wl, splat = _hidden_fixture(kind)
    o = run_oracle(wl)
    p = 8 * 16 + 8
    assert o["fwd"]["last"][p] == wl.n
    flips = oracle.flip_table([(p, splat, typ)])
    g = _fake(o, flips)
    assert np.abs(g["out"] - o["fwd"]["out"]).max() <= FWD_TOL and np.array_equal(g["last"], o["fwd"]["last"])
    ref = o["bwd"]["grad"][splat]
    moved = np.abs(g["grad"][splat].astype(np.float64) - ref)
    assert np.any(moved > 2 * (1e-4 + 1e-4 * np.abs(ref)))   # beyond the gradient tolerance without the flip
    fs = check_forward(g, o)
    assert fs["flipped_px"] == 0             # nothing to see in the forward
    bs = check_backward(g, o)
    assert bs["hidden_flips"] == 1
    g["grad"] = g["grad"].copy()
    g["grad"][splat, 8] += np.float32(2e-3)
    with pytest.raises(AssertionError):
        check_backward(g, o)


def test_a_flip_outside_the_uncertainty_is_refused():
    wl, _ = _hidden_fixture("clamp")
    o = run_oracle(wl)
    far = oracle.flip_table([(8 * 16 + 8, 1, oracle.DEC_ALPHA)])     # splat 1: alpha far above the cut
    f = oracle.forward_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, far, eps_alpha=EPS_ALPHA)
    assert f["refused"] == 1
    assert np.array_equal(f["out"], o["fwd"]["out"]) and np.array_equal(f["last"], o["fwd"]["last"])
