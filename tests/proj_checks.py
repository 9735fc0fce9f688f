"""Comparison of a float32 projection (forward and backward) with the double
oracle, with tolerances derived from the arithmetic.

Both sides read the same float32 Gaussians and float32-exact camera, so the
only differences are the float32 roundings of the implementation under test
(u = 2^-24 per operation).  First-order forward error bounds, each with a
safety factor of 4 or more over the operation count:

- camera-space p = W mu + t: |dp_i| <= 4u A_i, A_i = sum_j |W_ij mu_j| + |t_i|;
- pixel mean: |d mean_x| <= 16u (fx/z A_0 + fx |x| / z^2 A_2 + |fx x / z| + |cx|),
  likewise for y; depth: 8u A_2;
- conic: measured in its own metric, delta = || Q^-1/2 (Q' - Q) Q^-1/2 ||_2 =
  max |eigenvalue of Sigma2 (Q' - Q)|, which bounds the relative change of
  sigma = 1/2 d^T Q d at every pixel.  Each entry of Sigma2 = V V^T + eps I is
  a dot product with relative error ~3u, which in this metric is up to
  ~3u tr(Sigma2) / lambda_min(Sigma2); an error of p feeds J at relative
  kappa_p = (A_0 + A_1 + A_2) / z.  Tolerance 32u (1 + kappa_p + tr / lambda_min);
- color_a = 1 / (1 + exp(-logit)): 8u color_a (exp within 2 ulp);
- rgb: copied, bit-exact;
- gradients: dL/dtheta_k = sum_j G_j dsplat_j/dtheta_k.  The partials of the
  conic carry the conic's relative error, those of the mean and color_a that
  of p, so |dg_k| <= 64u [(1 + kappa_p) (|G_mean| J_mean,k + |G_alpha| J_alpha,k)
  + (1 + kappa_p + tr / lambda_min) |G_conic| J_conic,k], with J_group,k the
  largest magnitude of the partials of that group of splat fields, taken
  from central differences of the double oracle, and |G_group| the sum of
  |G_j| over the group.  Where the last sum of a gradient cancels (the
  rotation gradient of an isotropic Gaussian is exactly 0, a sum of terms that
  are not), its rounding scales with the sum of |terms| instead, which the
  oracle reports (gabs): + 16u (1 + kappa_p + tr / lambda_min) gabs_k.

A Gaussian is visible on both sides or on neither, except within 8u A_2 of
the near plane (the pages give no near plane; none of the scenes puts a mean
there).  Invisible Gaussians must give exact zeros.
"""
import numpy as np

import oracle

U = 2.0 ** -24


def _abs_p(g, cam):
    W = cam[:9].reshape(3, 3)
    t = cam[9:12]
    mu = g[:, 0:3]
    return np.abs(mu) @ np.abs(W).T + np.abs(t)        # [n, 3]: A_i


def _sigma2_from_conic(sp):
    a, b, c = sp[:, 2], sp[:, 3], sp[:, 4]
    det = a * c - b * b
    s00, s01, s11 = c / det, -b / det, a / det
    tr = s00 + s11
    disc = np.sqrt(np.maximum(0.25 * tr * tr - (s00 * s11 - s01 * s01), 0.0))
    return s00, s01, s11, tr, 0.5 * tr - disc


def conic_delta(sp_test, sp_ref):
    """delta = max |eigenvalue| of Sigma2_ref (Q_test - Q_ref), per row."""
    s00, s01, s11, _, _ = _sigma2_from_conic(sp_ref)
    da = sp_test[:, 2] - sp_ref[:, 2]
    db = sp_test[:, 3] - sp_ref[:, 3]
    dc = sp_test[:, 4] - sp_ref[:, 4]
    m00 = s00 * da + s01 * db
    m01 = s00 * db + s01 * dc
    m10 = s01 * da + s11 * db
    m11 = s01 * db + s11 * dc
    tr = m00 + m11
    det = m00 * m11 - m01 * m10
    disc = np.sqrt(np.maximum(0.25 * tr * tr - det, 0.0))
    return np.maximum(np.abs(0.5 * tr + disc), np.abs(0.5 * tr - disc))


def _conditioning(g64, cam, sp_ref, depth_ref):
    A = _abs_p(g64, cam)
    z = np.where(depth_ref > 0, depth_ref, 1.0)
    kappa_p = A.sum(axis=1) / z
    _, _, _, tr, lmin = _sigma2_from_conic(sp_ref)
    return A, z, 1.0 + kappa_p + tr / lmin


@np.errstate(all="ignore")
def check_forward(g32, cam, sp, depth):
    """Compares float32 splats [n, 9] and depths [n] with the oracle."""
    g64 = g32.astype(np.float64)
    sp = np.asarray(sp, dtype=np.float64)
    depth = np.asarray(depth, dtype=np.float64)
    sp_ref, d_ref, vis = oracle.project_forward(g64, cam)
    assert np.array_equal(sp[:, 5:8], g32[:, 11:14].astype(np.float64), equal_nan=True), "rgb not copied"
    A, z, cond = _conditioning(np.nan_to_num(g64), cam, np.where(vis[:, None], sp_ref, 1.0), d_ref)
    vis_test = sp[:, 2] > 0
    knife = np.abs(np.where(np.isfinite(g64).all(axis=1), d_ref, 0) - cam[16]) <= 8 * U * A[:, 2]
    assert np.all((vis_test == vis) | knife), f"visibility differs at {np.nonzero(vis_test != vis)[0][:8]}"
    inv = ~vis & ~knife
    assert np.all(sp[inv][:, [0, 1, 2, 3, 4, 8]] == 0) and np.all(depth[inv] == 0), "invisible not zero"
    v = vis & vis_test
    fx, fy, cx, cy = cam[12], cam[13], cam[14], cam[15]
    xr = sp_ref[:, 0] - cx
    yr = sp_ref[:, 1] - cy
    tol_x = 16 * U * (fx / z * A[:, 0] + np.abs(xr) / z * A[:, 2] + np.abs(xr) + abs(cx))
    tol_y = 16 * U * (fy / z * A[:, 1] + np.abs(yr) / z * A[:, 2] + np.abs(yr) + abs(cy))
    ex = np.abs(sp[:, 0] - sp_ref[:, 0])
    ey = np.abs(sp[:, 1] - sp_ref[:, 1])
    ed = np.abs(depth - d_ref)
    delta = conic_delta(sp, sp_ref)
    ea = np.abs(sp[:, 8] - sp_ref[:, 8])
    checks = {
        "mean_x": (ex, tol_x), "mean_y": (ey, tol_y), "depth": (ed, 8 * U * A[:, 2]),
        "conic": (delta, 32 * U * cond), "color_a": (ea, 8 * U * sp_ref[:, 8]),
    }
    stats = {"visible": int(v.sum()), "invisible": int((~vis).sum()), "knife": int(knife.sum())}
    for name, (err, tol) in checks.items():
        bad = v & ~(err <= tol)
        assert not bad.any(), (f"{name}: {bad.sum()} Gaussians beyond tolerance, first "
                               f"{np.nonzero(bad)[0][:5]} err {err[bad][:5]} tol {tol[bad][:5]}")
        stats[name + "_max_err_over_tol"] = float(np.max(err[v] / tol[v])) if v.any() else 0.0
    return stats


def partial_scales(g64, cam, vis, rel_h=1e-6):
    """Magnitudes [n, 14] x 3 of the partials of the mean (max over x, y), the
    conic (max over a, b, c) and color_a with respect to each Gaussian field, by
    central differences of the oracle forward."""
    n = g64.shape[0]
    out = np.zeros((3, n, 14))
    gv = np.where(vis[:, None], g64, 0.0)
    for k in range(14):
        h = rel_h * np.maximum(1.0, np.abs(gv[:, k]))
        gp, gm = gv.copy(), gv.copy()
        gp[:, k] += h
        gm[:, k] -= h
        sp_p, _, _ = oracle.project_forward(gp, cam)
        sp_m, _, _ = oracle.project_forward(gm, cam)
        d = np.abs(sp_p - sp_m) / (2 * h[:, None])
        out[0, :, k] = d[:, 0:2].max(axis=1)
        out[1, :, k] = d[:, 2:5].max(axis=1)
        out[2, :, k] = d[:, 8]
    return out


@np.errstate(all="ignore")
def backward_tolerance(g64, cam, G64, extra_G=None):
    """Per-element tolerance [n, 14] of a float32 projection backward, and the
    oracle's gradient and visibility.  extra_G: an uncertainty [n, 9] of G
    itself (for example a rasterizer gradient's tolerance), propagated through
    the same partial magnitudes."""
    sp_ref, d_ref, vis = oracle.project_forward(g64, cam)
    ref, gabs = oracle.project_backward(g64, cam, G64, with_abs=True)
    A, z, cond = _conditioning(np.nan_to_num(g64), cam, np.where(vis[:, None], sp_ref, 1.0), d_ref)
    kappa = 1.0 + A.sum(axis=1) / z
    J = partial_scales(g64, cam, vis)

    def spread(G, w_mean, w_conic):
        aG = np.abs(G)
        return (w_mean[:, None] * ((aG[:, 0] + aG[:, 1])[:, None] * J[0] + aG[:, 8][:, None] * J[2])
                + w_conic[:, None] * (aG[:, 2] + aG[:, 3] + aG[:, 4])[:, None] * J[1])

    tol = U * (64 * spread(G64, kappa, cond) + 16 * cond[:, None] * gabs)
    if extra_G is not None:
        ones = np.ones_like(cond)
        tol = tol + spread(extra_G, ones, ones)
        tol[:, 11:14] += extra_G[:, 5:8]
    return ref, tol, vis


def check_backward(g32, cam, G32, grad, extra_G=None):
    g64 = g32.astype(np.float64)
    G64 = np.asarray(G32, dtype=np.float64)
    grad = np.asarray(grad, dtype=np.float64)
    ref, tol, vis = backward_tolerance(g64, cam, G64, extra_G)
    assert np.all(grad[~vis] == 0), "an invisible Gaussian got a gradient"
    if extra_G is None:
        assert np.array_equal(grad[vis][:, 11:14], G64[vis][:, 5:8]), "rgb gradient not copied"
    err = np.abs(grad - ref)
    bad = vis[:, None] & ~(err <= tol + 1e-30)
    assert not bad.any(), (f"{bad.any(axis=1).sum()} Gaussians' gradients beyond tolerance; first "
                           f"(row, field) {np.argwhere(bad)[:5].tolist()} err {err[bad][:5]} tol {tol[bad][:5]}")
    ratio = err[vis] / (tol[vis] + 1e-30)
    return {"visible": int(vis.sum()), "max_err_over_tol": float(ratio.max()) if vis.any() else 0.0}
