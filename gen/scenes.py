"""Seeded synthetic 3-D Gaussian scenes and pinhole cameras.

Inputs of the projection step only: this module draws Gaussians and places a
camera; it computes no projection, conic or sigmoid.  Both the oracle tests
and the CUDA path take their inputs from here.

A Gaussian is 14 float32 values:
    mean xyz, log_scale xyz, quat wxyz (not normalised), logit_opacity, rgb
A camera is 18 values, every one exactly representable in float32:
    W row-major (world -> camera rotation), t, fx, fy, cx, cy, z_near, eps
with camera-space p = W x + t, x right, y down, z forward (depth).

The Lego-shaped scene stands in for the pages' trained Lego model
("forward/adam audit": 800x800 views, ~407k Gaussians at the final
checkpoint; "A.9 f16 forward": 83,734 in the sh3 run).  The NeRF-synthetic
views it imitates sit on a sphere of radius ~4 around an object inside
[-1.2, 1.2]^3, with a horizontal field of view of 0.6911 rad.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GAUSSIAN_FIELDS = ("mean_x", "mean_y", "mean_z", "log_scale_x", "log_scale_y", "log_scale_z",
                   "quat_w", "quat_x", "quat_y", "quat_z", "logit_opacity", "r", "g", "b")


@dataclass
class Scene:
    name: str
    width: int
    height: int
    gaussians: np.ndarray       # float32 [N, 14]
    camera: np.ndarray          # float64 [18], float32-exact values
    dl_dsplat: np.ndarray       # float32 [N, 9], N(0, 1)
    recipe: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.gaussians.shape[0])


def look_at_camera(eye, target, up, fx, fy, cx, cy, z_near=0.01, eps=0.3) -> np.ndarray:
    """Camera at `eye` looking at `target`, y axis pointing away from `up`.
    Rounded to float32 so that both sides of a comparison see the same numbers."""
    eye = np.asarray(eye, dtype=np.float64)
    fwd = np.asarray(target, dtype=np.float64) - eye
    fwd /= np.linalg.norm(fwd)
    right = np.cross(fwd, np.asarray(up, dtype=np.float64))
    right /= np.linalg.norm(right)
    down = np.cross(fwd, right)
    W = np.stack([right, down, fwd]).astype(np.float32).astype(np.float64)
    t = (-(W @ eye)).astype(np.float32).astype(np.float64)
    cam = np.concatenate([W.ravel(), t, [fx, fy, cx, cy, z_near, eps]])
    return cam.astype(np.float32).astype(np.float64)


def _logit(p):
    return np.log(p) - np.log1p(-p)


def lego_scene(n: int = 409_660, seed: int = 3, tail: float = 0.76, name: str = "lego_scene") -> Scene:
    """Gaussians of a Lego-shaped model seen from one NeRF-synthetic-like view.

    Means: 8-component isotropic GMM, centres U[-0.6, 0.6]^3, component std
    U(0.15, 0.45), clipped to [-1.2, 1.2]^3.  Log-scales i.i.d. N(ln 0.009, 1.0)
    per axis, clipped to [ln 2.7e-4, ln 0.72] (about 0.3 to 200 px at depth 4).
    Quaternions N(0, 1)^4.  Opacity logits N(0.5, 1.5), with a `tail` fraction
    at opacity U(0, 0.01) (the same low-opacity share as the 2-D Lego-shaped set).
    rgb U(0, 1).  Camera: 800x800, fx = fy = 400 / tan(0.6911 / 2), radius 4.03,
    azimuth 30 deg, elevation 30 deg, z up, looking at the origin.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    k = 8
    centres = rng.uniform(-0.6, 0.6, size=(k, 3))
    comp_std = rng.uniform(0.15, 0.45, size=k)
    comp = rng.integers(0, k, size=n)
    means = np.clip(centres[comp] + rng.standard_normal((n, 3)) * comp_std[comp][:, None], -1.2, 1.2)
    log_scale = np.clip(rng.normal(np.log(0.009), 1.0, size=(n, 3)), np.log(2.7e-4), np.log(0.72))
    quat = rng.standard_normal((n, 4))
    logit = rng.normal(0.5, 1.5, size=n)
    rgb = rng.uniform(0.0, 1.0, size=(n, 3))
    if tail > 0.0:
        low = rng.permutation(n)[: int(round(tail * n))]
        logit[low] = _logit(rng.uniform(1e-6, 0.01, size=low.size))
    g = np.concatenate([means, log_scale, quat, logit[:, None], rgb], axis=1).astype(np.float32)
    dl = rng.standard_normal((n, 9)).astype(np.float32)
    w = h = 800
    f = 400.0 / np.tan(0.6911 / 2.0)
    az, el, r = np.radians(30.0), np.radians(30.0), 4.03
    eye = r * np.array([np.cos(el) * np.cos(az), np.cos(el) * np.sin(az), np.sin(el)])
    cam = look_at_camera(eye, (0.0, 0.0, 0.0), (0.0, 0.0, 1.0), f, f, 399.5, 399.5)
    return Scene(name, w, h, g, cam, dl,
                 {"seed": seed, "gmm_components": k, "log_scale": "N(ln0.009,1.0) clip",
                  "low_opacity_fraction": tail, "fx": float(cam[12])})


def edge_scene(seed: int = 11) -> Scene:
    """Gaussians that exercise every visibility rule, each kind in a block of 16:
    in front of the camera (visible), behind it, between the camera and the
    near plane, zero quaternion, NaN and +inf in one field each, needle-thin
    (scale ratio up to 1e4) and very large (200 px) splats, and means far
    off-screen but in front of the camera."""
    rng = np.random.Generator(np.random.PCG64(seed))
    m = 16
    cam = look_at_camera((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), (0.0, -1.0, 0.0), 1000.0, 1000.0, 255.5, 255.5)

    def block(means, log_scale=None):
        q = rng.standard_normal((m, 4))
        ls = np.log(0.02) + 0.3 * rng.standard_normal((m, 3)) if log_scale is None else log_scale
        lo = rng.normal(0.0, 1.5, size=(m, 1))
        rgb = rng.uniform(0, 1, size=(m, 3))
        return np.concatenate([means, ls, q, lo, rgb], axis=1)

    front = block(rng.uniform(-0.5, 0.5, (m, 3)))
    behind = block(np.column_stack([rng.uniform(-0.5, 0.5, (m, 2)), rng.uniform(-9.0, -4.5, m)]))
    near = block(np.column_stack([rng.uniform(-1e-3, 1e-3, (m, 2)), rng.uniform(-4.0, -3.995, m)]))
    zero_q = block(rng.uniform(-0.5, 0.5, (m, 3)))
    zero_q[:, 6:10] = 0.0
    nan = block(rng.uniform(-0.5, 0.5, (m, 3)))
    nan[np.arange(m), rng.integers(0, 14, m)] = np.nan
    inf = block(rng.uniform(-0.5, 0.5, (m, 3)))
    inf[np.arange(m), rng.integers(0, 14, m)] = np.inf
    needle_ls = np.column_stack([rng.uniform(np.log(0.05), np.log(0.5), m),
                                 rng.uniform(np.log(5e-5), np.log(5e-4), m),
                                 rng.uniform(np.log(5e-5), np.log(5e-4), m)])
    needle = block(rng.uniform(-0.5, 0.5, (m, 3)), needle_ls)
    large = block(rng.uniform(-0.5, 0.5, (m, 3)), np.full((m, 3), np.log(0.8)))
    off = block(np.column_stack([rng.uniform(-30.0, 30.0, (m, 2)), rng.uniform(2.0, 6.0, m)]))
    g = np.concatenate([front, behind, near, zero_q, nan, inf, needle, large, off]).astype(np.float32)
    dl = rng.standard_normal((g.shape[0], 9)).astype(np.float32)
    return Scene("edge_scene", 512, 512, g, cam, dl, {"seed": seed, "block": m})


def random_scene(seed: int) -> Scene:
    """A randomised projection case: 1..5,000 Gaussians in a box of side 4
    around the origin, log-scales N(ln 0.05, 1.2) per axis, any rotation and
    logit; a look-at camera at distance U(0.5, 8) (so some Gaussians fall behind
    it or inside its near plane), focal lengths U(100, 2000) and a principal
    point anywhere in a 64..1024-pixel image, dilation 0.3 or 0."""
    rng = np.random.Generator(np.random.PCG64(2_000_003 + seed))
    n = int(rng.integers(1, 5001))
    means = rng.uniform(-2.0, 2.0, (n, 3))
    log_scale = rng.normal(np.log(0.05), 1.2, (n, 3))
    quat = rng.standard_normal((n, 4))
    logit = rng.normal(0.0, 2.0, n)
    rgb = rng.uniform(0.0, 1.0, (n, 3))
    g = np.concatenate([means, log_scale, quat, logit[:, None], rgb], axis=1).astype(np.float32)
    w, h = (int(v) for v in rng.integers(64, 1025, 2))
    d = rng.uniform(0.5, 8.0)
    direction = rng.standard_normal(3)
    direction /= np.linalg.norm(direction)
    up = np.array([0.0, 0.0, 1.0]) if abs(direction[2]) < 0.9 else np.array([1.0, 0.0, 0.0])
    f = rng.uniform(100.0, 2000.0, 2)
    cam = look_at_camera(d * direction, (0.0, 0.0, 0.0), up, f[0], f[1], rng.uniform(0, w), rng.uniform(0, h),
                         eps=0.3 if seed % 3 else 0.0)
    dl = rng.standard_normal((n, 9)).astype(np.float32)
    return Scene(f"random_scene{seed}", w, h, g, cam, dl, {"seed": seed})
