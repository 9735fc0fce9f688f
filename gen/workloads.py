"""Seeded synthetic Splat2D workloads.

This module only draws random inputs; it holds none of the rasterizer's
arithmetic (no tile rectangles, no compositing, no key packing).  Both the
CPU oracle tests and the CUDA path take their inputs from here.

Workload shapes follow the pages' Lego scene ("p3-forward-adam-audit": 800x800
image, 2,500 16x16 tiles, ~407k splats and ~970k tile pairs at the final
checkpoint; "a-9-f16-forward-negative": 83,734 splats for the sh3 run;
"p2-w1-warp-sparse-skip" body: ~94% of splat-pixel evaluations contribute
nothing).  The Lego checkpoints themselves are not available, so these seeded
distributions stand in for them.

A Splat2D record is 9 float32 values in this order:
    mean_x, mean_y, conic_a, conic_b, conic_c, color_r, color_g, color_b, color_a
with the conic (a, b, c) the inverse of the 2-D covariance, i.e.
sigma(d) = 1/2 (a dx^2 + c dy^2) + b dx dy is half the squared Mahalanobis
distance.  Depths are a separate float32 array.  dL/dout is a float4 per
pixel (rgb drawn N(0,1), w zero).

Draw order inside one workload is fixed: means, depths, principal stds,
rotation, rgb, opacity, then config-specific subsets, then dL/dout last.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SPLAT_FIELDS = ("mean_x", "mean_y", "conic_a", "conic_b", "conic_c",
                "color_r", "color_g", "color_b", "color_a")


@dataclass
class Workload:
    name: str
    width: int
    height: int
    splats: np.ndarray          # float32 [N, 9]
    depths: np.ndarray          # float32 [N]
    dl_dout: np.ndarray         # float32 [H*W, 4], w == 0
    recipe: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.splats.shape[0])


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _conics(s1, s2, theta):
    """Inverse of R diag(s1^2, s2^2) R^T, in float64, returned as (a, b, c)."""
    ct, st = np.cos(theta), np.sin(theta)
    v1, v2 = s1 * s1, s2 * s2
    sxx = ct * ct * v1 + st * st * v2
    syy = st * st * v1 + ct * ct * v2
    sxy = ct * st * (v1 - v2)
    det = sxx * syy - sxy * sxy
    return syy / det, -sxy / det, sxx / det


def _gmm_means(rng, n, k, lo_xy, hi_xy, comp_std_lo, comp_std_hi, width, height):
    centres = rng.uniform(lo_xy, hi_xy, size=(k, 2))
    comp_std = rng.uniform(comp_std_lo, comp_std_hi, size=k)
    comp = rng.integers(0, k, size=n)
    xy = centres[comp] + rng.standard_normal((n, 2)) * comp_std[comp][:, None]
    xy[:, 0] = np.clip(xy[:, 0], 0.0, np.nextafter(float(width), 0.0))
    xy[:, 1] = np.clip(xy[:, 1], 0.0, np.nextafter(float(height), 0.0))
    return xy


def _assemble(name, rng, width, height, means, depths, s1, s2, theta, rgb, opac, recipe):
    a, b, c = _conics(s1, s2, theta)
    n = means.shape[0]
    sp = np.empty((n, 9), dtype=np.float32)
    sp[:, 0:2] = means
    sp[:, 2] = a
    sp[:, 3] = b
    sp[:, 4] = c
    sp[:, 5:8] = rgb
    sp[:, 8] = opac
    dl = np.zeros((width * height, 4), dtype=np.float32)
    dl[:, 0:3] = rng.standard_normal((width * height, 3))
    return Workload(name, width, height, sp, depths.astype(np.float32), dl, recipe)


# Low-opacity tail for the final Lego-shaped set: this fraction of splats gets
# color_a ~ U(0, 0.01).  Chosen so that the oracle-measured share of
# non-contributing splat-pixel evaluations lands near the pages' 94%
# (checked by tests/test_workloads.py).
LEGO_FINAL_TAIL = 0.76
# Common factor applied to the long-axis std of the 5% "large" splats of the
# stress set.  Unscaled they would emit ~74M tile pairs; at 0.25 the set emits
# ~24M (the base std distribution alone already emits ~18M).
STRESS_LARGE_SCALE = 0.25


def tiny(seed: int = 0) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    n, w, h = 256, 64, 64
    means = rng.uniform(0.0, 64.0, size=(n, 2))
    depths = rng.uniform(1.0, 10.0, size=n)
    s = rng.lognormal(np.log(3.0), 0.5, size=(n, 2))
    theta = rng.uniform(0.0, np.pi, size=n)
    rgb = rng.uniform(0.0, 1.0, size=(n, 3))
    opac = _sigmoid(rng.standard_normal(n))
    return _assemble("tiny", rng, w, h, means, depths, s[:, 0], s[:, 1], theta, rgb, opac,
                     {"seed": seed, "std": "LN(ln3,0.5)"})


def small(seed: int = 1) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    n, w, h = 10_000, 256, 256
    means = rng.uniform(0.0, 256.0, size=(n, 2))
    depths = rng.uniform(1.0, 10.0, size=n)
    s = rng.lognormal(np.log(4.0), 0.7, size=(n, 2))
    theta = rng.uniform(0.0, np.pi, size=n)
    rgb = rng.uniform(0.0, 1.0, size=(n, 3))
    opac = _sigmoid(rng.standard_normal(n))
    low = rng.permutation(n)[: int(round(0.15 * n))]
    opac[low] = rng.uniform(0.0, 0.01, size=low.size)
    return _assemble("small", rng, w, h, means, depths, s[:, 0], s[:, 1], theta, rgb, opac,
                     {"seed": seed, "std": "LN(ln4,0.7)", "low_opacity_fraction": 0.15})


def _lego(name, seed, n, std_mu, std_sigma, tail):
    rng = np.random.Generator(np.random.PCG64(seed))
    w = h = 800
    means = _gmm_means(rng, n, 8, 200.0, 600.0, 40.0, 120.0, w, h)
    depths = rng.uniform(2.0, 6.0, size=n)
    s = np.clip(rng.lognormal(np.log(std_mu), std_sigma, size=(n, 2)), 0.3, 200.0)
    theta = rng.uniform(0.0, np.pi, size=n)
    rgb = rng.uniform(0.0, 1.0, size=(n, 3))
    opac = _sigmoid(rng.normal(0.5, 1.5, size=n))
    recipe = {"seed": seed, "gmm_components": 8, "std": f"LN(ln{std_mu},{std_sigma}) clip[0.3,200]"}
    if tail > 0.0:
        low = rng.permutation(n)[: int(round(tail * n))]
        opac[low] = rng.uniform(0.0, 0.01, size=low.size)
        recipe["low_opacity_fraction"] = tail
    return _assemble(name, rng, w, h, means, depths, s[:, 0], s[:, 1], theta, rgb, opac, recipe)


def lego_early(seed: int = 2) -> Workload:
    return _lego("lego_early", seed, 83_734, 6.0, 0.9, 0.0)


def lego_final(seed: int = 3) -> Workload:
    return _lego("lego_final", seed, 409_660, 2.5, 1.0, LEGO_FINAL_TAIL)


def lego_pages(seed: int = 3) -> Workload:
    """lego_final's splat count and opacity mix at the pages' pair density:
    their final checkpoint binned 969,838 pairs for 407,267 splats (2.38 per
    splat); smaller footprints, std LN(ln 1.15, 0.6), give 983,065 pairs for
    409,660 splats (2.40 per splat)."""
    return _lego("lego_pages", seed, 409_660, 1.15, 0.6, LEGO_FINAL_TAIL)


def stress(seed: int = 4) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    n, w, h = 1_000_000, 1920, 1080
    means = _gmm_means(rng, n, 32, np.array([0.0, 0.0]), np.array([1920.0, 1080.0]),
                       60.0, 240.0, w, h)
    depths = rng.uniform(2.0, 6.0, size=n)
    s = np.clip(rng.lognormal(np.log(3.0), 1.2, size=(n, 2)), 0.3, 400.0)
    theta = rng.uniform(0.0, np.pi, size=n)
    rgb = rng.uniform(0.0, 1.0, size=(n, 3))
    opac = _sigmoid(rng.normal(0.5, 1.5, size=n))
    large = rng.permutation(n)[: int(round(0.05 * n))]
    s[large, 0] = np.exp(rng.uniform(np.log(50.0), np.log(400.0), size=large.size)) * STRESS_LARGE_SCALE
    return _assemble("stress", rng, w, h, means, depths, s[:, 0], s[:, 1], theta, rgb, opac,
                     {"seed": seed, "gmm_components": 32, "large_fraction": 0.05,
                      "large_scale": STRESS_LARGE_SCALE})


def lego_far(seed: int = 3, distance: float = 4.0) -> Workload:
    """lego_final seen from `distance` times farther away: a pinhole camera
    maps a Gaussian's footprint linearly in 1/depth, so the means move toward
    the image centre, every std shrinks by that factor (the conic grows by its
    square) and depths grow by it.  The whole object lands in a few dozen tiles
    with very long lists, the crowded-tile case the frame's other sets lack."""
    base = lego_final(seed)
    sp = base.splats.astype(np.float64)
    c = (base.width - 1) / 2.0
    sp[:, 0:2] = c + (sp[:, 0:2] - c) / distance
    sp[:, 2:5] *= distance ** 2
    recipe = dict(base.recipe, name_of_base="lego_final", distance=distance)
    return Workload("lego_far", base.width, base.height, sp.astype(np.float32),
                    (base.depths.astype(np.float64) * distance).astype(np.float32), base.dl_dout, recipe)


CONFIGS = {
    "tiny": tiny,
    "small": small,
    "lego_early": lego_early,
    "lego_final": lego_final,
    "stress": stress,
    "lego_far": lego_far,
    "lego_pages": lego_pages,
}


def make(name: str) -> Workload:
    return CONFIGS[name]()


def overlap_fixture(size: int, n: int = 24, seed: int = 7) -> Workload:
    """n splats piled near the centre of a size x size image (all overlap).

    Mirrors the pages' 24-splat overlap fixtures at 32x32 (no out-of-bounds
    pixels) and 24x24 (out-of-bounds pixels in the partial tiles)
    ("p3-per-splat-backward", section 2).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    means = size * 0.5 + rng.uniform(-size * 0.25, size * 0.25, size=(n, 2))
    depths = rng.uniform(1.0, 5.0, size=n)
    s = rng.uniform(2.0, size * 0.3, size=(n, 2))
    theta = rng.uniform(0.0, np.pi, size=n)
    rgb = rng.uniform(0.0, 1.0, size=(n, 3))
    opac = rng.uniform(0.2, 0.9, size=n)
    return _assemble(f"overlap{size}", rng, size, size, means, depths, s[:, 0], s[:, 1], theta, rgb,
                     opac, {"seed": seed})


def from_arrays(name, width, height, splats, depths, dl_dout=None, seed=0) -> Workload:
    sp = np.ascontiguousarray(splats, dtype=np.float32).reshape(-1, 9)
    dp = np.ascontiguousarray(depths, dtype=np.float32).reshape(-1)
    if dl_dout is None:
        rng = np.random.Generator(np.random.PCG64(seed))
        dl_dout = np.zeros((width * height, 4), dtype=np.float32)
        dl_dout[:, 0:3] = rng.standard_normal((width * height, 3))
    return Workload(name, width, height, sp, dp, np.ascontiguousarray(dl_dout, dtype=np.float32))


def elongated_fixture(seed: int = 8, n: int = 3000, size: int = 512) -> Workload:
    """Thin, rotated splats of every size, some centred off-image.

    Long-axis std log-uniform in [2, 150] px, aspect ratio log-uniform in
    [1, 400], any orientation, a third of the splats at color_a in (0, 0.01)
    so their alpha >= 1/255 ellipse is much smaller than their 3-sigma box.
    Exercises the culling of staged splats against pixel blocks.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    means = rng.uniform(-0.2 * size, 1.2 * size, size=(n, 2))
    depths = rng.uniform(1.0, 8.0, size=n)
    s_long = np.exp(rng.uniform(np.log(2.0), np.log(150.0), size=n))
    aspect = np.exp(rng.uniform(0.0, np.log(400.0), size=n))
    s_short = np.maximum(s_long / aspect, 0.05)
    theta = rng.uniform(0.0, np.pi, size=n)
    rgb = rng.uniform(0.0, 1.0, size=(n, 3))
    opac = _sigmoid(rng.normal(0.5, 1.5, size=n))
    low = rng.permutation(n)[: n // 3]
    opac[low] = rng.uniform(0.0, 0.01, size=low.size)
    return _assemble("elongated", rng, size, size, means, depths, s_long, s_short, theta, rgb, opac,
                     {"seed": seed, "aspect": "logU(1,400)", "long_std": "logU(2,150)"})



def random_case(seed: int) -> Workload:
    """A randomised small case for fuzzing: image sides 1..300 (rarely a
    multiple of 16), 0..3,000 splats centred anywhere from 50 px outside the
    image to inside it, stds log-uniform in [0.2, 80] px with aspect ratios to
    100, color_a in (0, 1) (the rasterizer's domain), depths U(0.5, 20) with a few exact ties; 2% of the
    splats get a culled value (depth <= 0 or NaN, a NaN field, a negative
    determinant)."""
    rng = np.random.Generator(np.random.PCG64(1_000_003 + seed))
    w = int(rng.integers(1, 301))
    h = int(rng.integers(1, 301))
    n = int(rng.integers(0, 3001)) if seed % 7 else 0
    means = np.column_stack([rng.uniform(-50.0, w + 50.0, n), rng.uniform(-50.0, h + 50.0, n)])
    depths = rng.uniform(0.5, 20.0, n)
    ties = rng.random(n) < 0.1
    depths[ties] = np.round(depths[ties])
    s1 = np.exp(rng.uniform(np.log(0.2), np.log(80.0), n))
    s2 = s1 / np.exp(rng.uniform(0.0, np.log(100.0), n))
    theta = rng.uniform(0.0, np.pi, n)
    rgb = rng.uniform(0.0, 1.0, (n, 3))
    opac = rng.uniform(0.0, 1.0, n)
    wl = _assemble(f"random{seed}", rng, w, h, means, depths, np.maximum(s2, 0.05), s1, theta, rgb, opac,
                   {"seed": seed})
    bad = np.nonzero(rng.random(n) < 0.02)[0]
    for j, i in enumerate(bad):
        kind = j % 4
        if kind == 0:
            wl.depths[i] = -1.0 if j % 8 == 0 else 0.0
        elif kind == 1:
            wl.depths[i] = np.nan
        elif kind == 2:
            wl.splats[i, int(rng.integers(0, 9))] = np.nan
        else:
            wl.splats[i, 3] = np.sqrt(abs(wl.splats[i, 2] * wl.splats[i, 4])) * 1.5   # b^2 > a c
    return wl
