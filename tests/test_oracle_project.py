"""Pins of the projection oracle (oracle/project.c) to things other than itself.

- Closed form: an isotropic Gaussian on the optical axis of an axis-aligned
  camera projects to the principal point with conic 1 / ((f s / z)^2 + eps) on
  both axes and no cross term; color_a is the sigmoid of the logit.
- Invariances: scaling the quaternion changes nothing; rotating the world and
  the camera together (W -> W Q^T, mu -> Q mu, rotation -> Q R) changes
  nothing; a Gaussian behind the near plane is not visible and gets no
  gradient.
- A rotation by 90 degrees about the optical axis swaps the conic's a and c.
- The backward against central finite differences of the forward, for every
  one of the 14 parameters of random visible Gaussians.
"""
import numpy as np
import pytest

import oracle


def camera(W=np.eye(3), t=(0.0, 0.0, 0.0), fx=1000.0, fy=900.0, cx=399.5, cy=299.5, z_near=0.01, eps=0.3):
    return np.concatenate([np.asarray(W, dtype=np.float64).ravel(), np.asarray(t, dtype=np.float64),
                           [fx, fy, cx, cy, z_near, eps]])


def gaussian(mean=(0.0, 0.0, 4.0), log_scale=(np.log(0.05),) * 3, quat=(1.0, 0.0, 0.0, 0.0), logit=0.5,
             rgb=(0.2, 0.3, 0.4)):
    return np.concatenate([mean, log_scale, quat, [logit], rgb]).astype(np.float64)


def quat_of_rotation(axis, angle):
    axis = np.asarray(axis, dtype=np.float64) / np.linalg.norm(axis)
    return np.concatenate([[np.cos(angle / 2)], np.sin(angle / 2) * axis])


def rotation(q):
    w, x, y, z = np.asarray(q) / np.linalg.norm(q)
    return np.array([[1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)],
                     [2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)],
                     [2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)]])


def quat_mul(p, q):
    w1, x1, y1, z1 = p
    w2, x2, y2, z2 = q
    return np.array([w1 * w2 - x1 * x2 - y1 * y2 - z1 * z2, w1 * x2 + x1 * w2 + y1 * z2 - z1 * y2,
                     w1 * y2 - x1 * z2 + y1 * w2 + z1 * x2, w1 * z2 + x1 * y2 - y1 * x2 + z1 * w2])


def test_isotropic_gaussian_on_the_axis_closed_form():
    s, z, fx, fy, eps = 0.05, 4.0, 1000.0, 900.0, 0.3
    sp, d, vis = oracle.project_forward(gaussian(mean=(0, 0, z), log_scale=(np.log(s),) * 3),
                                        camera(fx=fx, fy=fy, eps=eps))
    assert vis[0] and d[0] == z
    assert sp[0, 0] == pytest.approx(399.5) and sp[0, 1] == pytest.approx(299.5)
    assert sp[0, 2] == pytest.approx(1.0 / ((fx * s / z) ** 2 + eps), rel=1e-14)
    assert sp[0, 4] == pytest.approx(1.0 / ((fy * s / z) ** 2 + eps), rel=1e-14)
    assert abs(sp[0, 3]) < 1e-18
    assert sp[0, 8] == pytest.approx(1.0 / (1.0 + np.exp(-0.5)), rel=1e-15)
    assert np.array_equal(sp[0, 5:8], [0.2, 0.3, 0.4])


def test_off_axis_mean_projects_by_pinhole():
    sp, d, _ = oracle.project_forward(gaussian(mean=(0.3, -0.2, 2.5)), camera(t=(0.1, 0.0, 0.5)))
    x, y, z = 0.4, -0.2, 3.0
    assert d[0] == pytest.approx(z)
    assert sp[0, 0] == pytest.approx(1000.0 * x / z + 399.5, rel=1e-14)
    assert sp[0, 1] == pytest.approx(900.0 * y / z + 299.5, rel=1e-14)


def test_anisotropic_axes_and_quarter_turn_swap_the_conic():
    g = gaussian(log_scale=(np.log(0.1), np.log(0.02), np.log(0.05)))
    cam = camera(fy=1000.0, eps=0.0)
    sp0, _, _ = oracle.project_forward(g, cam)
    f, z = 1000.0, 4.0
    assert sp0[0, 2] == pytest.approx((z / (f * 0.1)) ** 2, rel=1e-12)   # x axis: std 0.1
    assert sp0[0, 4] == pytest.approx((z / (f * 0.02)) ** 2, rel=1e-12)  # y axis: std 0.02
    g[6:10] = quat_of_rotation((0, 0, 1), np.pi / 2)
    sp1, _, _ = oracle.project_forward(g, cam)
    assert sp1[0, 2] == pytest.approx(sp0[0, 4], rel=1e-12)
    assert sp1[0, 4] == pytest.approx(sp0[0, 2], rel=1e-12)


def test_quaternion_scale_changes_nothing():
    rng = np.random.default_rng(3)
    g = gaussian(mean=(0.2, 0.1, 3.0), log_scale=(-2.0, -3.0, -2.5), quat=rng.normal(size=4))
    h = g.copy()
    h[6:10] *= 7.5
    a, _, _ = oracle.project_forward(g, camera())
    b, _, _ = oracle.project_forward(h, camera())
    assert np.allclose(a, b, rtol=1e-13, atol=0)


def test_rotating_world_and_camera_together_changes_nothing():
    rng = np.random.default_rng(4)
    g = gaussian(mean=(0.2, 0.1, 3.0), log_scale=(-2.0, -3.0, -2.5), quat=rng.normal(size=4))
    Wc = rotation(quat_of_rotation((0.3, 1.0, 0.2), 0.4))
    cam = camera(W=Wc, t=(0.1, -0.2, 0.3))
    qQ = quat_of_rotation((1.0, -0.5, 0.7), 1.1)
    Q = rotation(qQ)
    h = g.copy()
    h[0:3] = Q @ g[0:3]
    h[6:10] = quat_mul(qQ, g[6:10] / np.linalg.norm(g[6:10]))
    cam2 = camera(W=Wc @ Q.T, t=(0.1, -0.2, 0.3))
    a, da, _ = oracle.project_forward(g, cam)
    b, db, _ = oracle.project_forward(h, cam2)
    assert np.allclose(a, b, rtol=1e-10, atol=1e-12) and da[0] == pytest.approx(db[0], rel=1e-12)


def test_behind_the_near_plane_is_not_visible():
    g = np.stack([gaussian(mean=(0, 0, -1.0)), gaussian(mean=(0, 0, 0.005)), gaussian(mean=(0, 0, 2.0))])
    sp, d, vis = oracle.project_forward(g, camera())
    assert list(vis) == [False, False, True]
    assert np.all(sp[:2, [0, 1, 2, 3, 4, 8]] == 0) and np.all(d[:2] == 0)
    grad = oracle.project_backward(g, camera(), np.ones((3, 9)))
    assert np.all(grad[:2] == 0) and np.any(grad[2] != 0)


def test_backward_matches_central_differences():
    rng = np.random.default_rng(5)
    n = 12
    g = np.zeros((n, 14))
    g[:, 0:2] = rng.uniform(-0.8, 0.8, (n, 2))
    g[:, 2] = rng.uniform(2.0, 5.0, n)
    g[:, 3:6] = rng.uniform(np.log(0.01), np.log(0.2), (n, 3))
    g[:, 6:10] = rng.normal(size=(n, 4))
    g[:, 10] = rng.normal(0.0, 1.5, n)
    g[:, 11:14] = rng.uniform(0, 1, (n, 3))
    cam = camera(W=rotation(quat_of_rotation((0.2, 1.0, -0.3), 0.3)), t=(0.05, -0.1, 0.2))
    weights = rng.normal(size=(n, 9))
    grad = oracle.project_backward(g, cam, weights)

    def loss(gg):
        sp, _, _ = oracle.project_forward(gg, cam)
        return float(np.sum(weights * sp))

    for i in range(n):
        for k in range(14):
            h = 1e-6 * max(1.0, abs(g[i, k]))
            gp, gm = g.copy(), g.copy()
            gp[i, k] += h
            gm[i, k] -= h
            fd = (loss(gp) - loss(gm)) / (2 * h)
            assert grad[i, k] == pytest.approx(fd, rel=2e-5, abs=2e-5 * (1 + abs(fd))), (i, k)


def test_isotropic_gaussian_has_no_rotation_gradient():
    """An isotropic Gaussian looks the same under any rotation: the quaternion
    gradient vanishes (up to rounding of its terms, whose size gabs reports),
    and every |gradient| is at most its gabs."""
    rng = np.random.default_rng(6)
    g = np.stack([gaussian(mean=(0.3, -0.1, 3.0), log_scale=(np.log(0.07),) * 3, quat=rng.normal(size=4))
                  for _ in range(4)])
    grad, gabs = oracle.project_backward(g, camera(), rng.normal(size=(4, 9)), with_abs=True)
    assert np.all(gabs[:, 6:10] > 0)
    assert np.all(np.abs(grad[:, 6:10]) <= 1e-12 * gabs[:, 6:10])
    assert np.all(np.abs(grad) <= gabs * (1 + 1e-12))


def test_chain_rule_through_the_rasterizer():
    """d/dtheta of sum(dL/dout . render(project(theta))) by central differences
    of the double oracle (bins held fixed: they are piecewise constant) against
    the oracle's projection backward of its double rasterizer backward."""
    rng = np.random.default_rng(12)
    n, size = 30, 48
    g = np.zeros((n, 14))
    g[:, 0:2] = rng.uniform(-1.2, 1.2, (n, 2))
    g[:, 2] = rng.uniform(-0.5, 0.5, n)
    g[:, 3:6] = rng.uniform(np.log(0.15), np.log(0.5), (n, 3))
    g[:, 6:10] = rng.normal(size=(n, 4))
    g[:, 10] = rng.normal(0.0, 1.0, n)
    g[:, 11:14] = rng.uniform(0, 1, (n, 3))
    cam = camera(t=(0.0, 0.0, 4.0), fx=60.0, fy=60.0, cx=23.5, cy=23.5)
    dl = np.zeros((size * size, 4))
    dl[:, 0:3] = rng.normal(size=(size * size, 3))
    sp, d, vis = oracle.project_forward(g, cam)
    assert vis.all()
    _, idx, ranges = oracle.bin_splats(sp.astype(np.float32), d.astype(np.float32), size, size)
    b = oracle.backward(sp, idx, ranges, size, size, dl, f64=True)
    grad = oracle.project_backward(g, cam, b["grad"])

    def loss(gg):
        s2, _, _ = oracle.project_forward(gg, cam)
        out = oracle.forward(s2, idx, ranges, size, size, f64=True)["out"]
        return float(np.sum(out[:, 0:3] * dl[:, 0:3]))

    checked = 0
    for i in range(n):
        if b["knife"][i]:
            continue
        for k in (0, 1, 2, 3, 5, 6, 8, 10, 12):
            h = 1e-6 * max(1.0, abs(g[i, k]))
            gp, gm = g.copy(), g.copy()
            gp[i, k] += h
            gm[i, k] -= h
            fd = (loss(gp) - loss(gm)) / (2 * h)
            assert grad[i, k] == pytest.approx(fd, rel=1e-3, abs=1e-4 * (1 + abs(fd))), (i, k, grad[i, k], fd)
            checked += 1
    assert checked >= 100
