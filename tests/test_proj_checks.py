"""The projection comparison (tests/proj_checks.py) on the CPU: the oracle's own
result rounded to float32 passes, and mistakes planted in the oracle's inputs
or outputs are caught."""
import numpy as np
import pytest

import gen
import oracle
import proj_checks


@pytest.fixture(scope="module")
def scene():
    return gen.lego_scene(n=3000, seed=21)


def test_rounded_oracle_passes(scene):
    sp, d, _ = oracle.project_forward(scene.gaussians.astype(np.float64), scene.camera)
    st = proj_checks.check_forward(scene.gaussians, scene.camera, sp.astype(np.float32), d.astype(np.float32))
    assert st["visible"] == scene.n
    g = oracle.project_backward(scene.gaussians.astype(np.float64), scene.camera, scene.dl_dsplat)
    proj_checks.check_backward(scene.gaussians, scene.camera, scene.dl_dsplat, g.astype(np.float32))


def test_edge_scene_rounded_oracle_passes():
    e = gen.edge_scene()
    sp, d, vis = oracle.project_forward(e.gaussians.astype(np.float64), e.camera)
    st = proj_checks.check_forward(e.gaussians, e.camera, sp.astype(np.float32), d.astype(np.float32))
    assert st["invisible"] == int((~vis).sum()) == 5 * 16
    g = oracle.project_backward(e.gaussians.astype(np.float64), e.camera, e.dl_dsplat)
    proj_checks.check_backward(e.gaussians, e.camera, e.dl_dsplat, g.astype(np.float32))


@pytest.mark.parametrize("plant", ["eps", "mean", "focal", "alpha"])
def test_planted_forward_mistakes_are_caught(scene, plant):
    cam = scene.camera.copy()
    if plant == "eps":
        cam[17] *= 1.001
    if plant == "focal":
        cam[13] *= 1.0001
    sp, d, _ = oracle.project_forward(scene.gaussians.astype(np.float64), cam)
    if plant == "mean":
        sp[7, 0] += 1e-3
    if plant == "alpha":
        sp[9, 8] *= 1.0 + 1e-5
    with pytest.raises(AssertionError):
        proj_checks.check_forward(scene.gaussians, scene.camera, sp.astype(np.float32), d.astype(np.float32))


@pytest.mark.parametrize("field", [0, 2, 4, 7, 10, 12])
def test_planted_backward_mistakes_are_caught(scene, field):
    g64 = scene.gaussians.astype(np.float64)
    G = scene.dl_dsplat.astype(np.float64).copy()
    grad = oracle.project_backward(g64, scene.camera, G)
    grad[5, field] *= 1.0 + 1e-3
    with pytest.raises(AssertionError):
        proj_checks.check_backward(scene.gaussians, scene.camera, scene.dl_dsplat, grad.astype(np.float32))


def test_dropped_conic_term_is_caught(scene):
    g64 = scene.gaussians.astype(np.float64)
    G = scene.dl_dsplat.astype(np.float64).copy()
    G[:, 3] = 0.0                     # the gradient as if b did not depend on the Gaussian
    grad = oracle.project_backward(g64, scene.camera, G)
    with pytest.raises(AssertionError):
        proj_checks.check_backward(scene.gaussians, scene.camera, scene.dl_dsplat, grad.astype(np.float32))


@pytest.mark.parametrize("seed", range(6))
def test_rounded_oracle_passes_random_scenes(seed):
    sc = gen.random_scene(seed)
    g64 = sc.gaussians.astype(np.float64)
    sp, d, _ = oracle.project_forward(g64, sc.camera)
    proj_checks.check_forward(sc.gaussians, sc.camera, sp.astype(np.float32), d.astype(np.float32))
    g = oracle.project_backward(g64, sc.camera, sc.dl_dsplat)
    proj_checks.check_backward(sc.gaussians, sc.camera, sc.dl_dsplat, g.astype(np.float32))
