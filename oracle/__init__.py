"""Plain CPU oracle of the tile-binned 2-D splat rasterizer.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline leg use it; the product package never imports it.  The C source
(oracle.c, raster.inc) shares no code with the CUDA path.

Parity status: binning, forward and backward are pinned by
tests/test_oracle_pins.py (closed forms, brute force, the pages' printed
constants and pass counts, finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "raster.inc"),
        os.path.join(_HERE, "project.c"), os.path.join(_HERE, "oracle.h")]
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall", "-Wextra",
          "-shared", "-fPIC"]

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C, no GPU)."""
    newest = max(os.path.getmtime(p) for p in _SRC)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, os.path.join(_HERE, "oracle.c"),
                               os.path.join(_HERE, "project.c"), "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.orc_tile_rect.argtypes = [P, ctypes.c_float, i32, i32, P]
    lib.orc_tile_rect.restype = ctypes.c_int
    lib.orc_count_pairs.argtypes = [P, P, i32, i32, i32]
    lib.orc_count_pairs.restype = i64
    lib.orc_bin.argtypes = [P, P, i32, i32, i32, P, P, P, i64]
    lib.orc_bin.restype = i64
    lib.orc_radix_passes_4bit.argtypes = [ctypes.c_uint64]
    lib.orc_radix_passes_4bit.restype = i32
    for sfx in ("f32", "f64"):
        fw = getattr(lib, f"orc_forward_{sfx}")
        fw.argtypes = [P, P, P, i32, i32, P, P, P, P, f64, f64, P]
        fw.restype = None
        bw = getattr(lib, f"orc_backward_{sfx}")
        bw.argtypes = [P, i32, P, P, i32, i32, P, P, P, P, f64, f64, P]
        bw.restype = None
    for name in ("orc_forward_untiled_f32", "orc_forward_untiled_noskip_f32", "orc_forward_untiled_nobox_f32"):
        fn = getattr(lib, name)
        fn.argtypes = [P, P, i32, i32, i32, P, P, P]
        fn.restype = None
    lib.orc_forward_forced_f32.argtypes = [P, P, P, i32, i32, P, i64, P, P, P, f64, f64, P]
    lib.orc_forward_forced_f32.restype = None
    lib.orc_pixel_forced_f32.argtypes = [P, P, P, i32, i32, i32, i32, P, i64, f64, f64, P, P, P, i32, P, P]
    lib.orc_pixel_forced_f32.restype = None
    lib.orc_backward_forced_f32.argtypes = [P, i32, P, P, i32, i32, P, P, i64, P, P, f64, f64, P]
    lib.orc_backward_forced_f32.restype = None
    lib.orc_backward_targets_f32.argtypes = [P, i32, P, P, i32, i32, P, P, i64, P, i32, P, P, f64, f64, P]
    lib.orc_backward_targets_f32.restype = None
    lib.orc_splat_decisions_f32.argtypes = [P, i32, P, P, i32, i32, P, i64, ctypes.c_uint32, f64, f64, P, P,
                                            i32, P]
    lib.orc_splat_decisions_f32.restype = None
    lib.orc_pixel_backward_forced_f32.argtypes = [P, P, P, i32, i32, P, i32, i32, P, i64, ctypes.c_uint32, P,
                                                  f64, f64, P]
    lib.orc_pixel_backward_forced_f32.restype = None
    lib.orc_project_forward.argtypes = [P, i32, P, P, P, P]
    lib.orc_project_forward.restype = None
    lib.orc_project_backward.argtypes = [P, i32, P, P, P, P]
    lib.orc_project_backward.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def tiles(width: int, height: int):
    return (width + 15) // 16, (height + 15) // 16


def tile_rect(splat, depth, width, height):
    lib = _load()
    s = _f32(splat).reshape(9)
    r = np.zeros(4, dtype=np.int32)
    tx, ty = tiles(width, height)
    ok = lib.orc_tile_rect(_ptr(s), ctypes.c_float(depth), tx, ty, _ptr(r))
    return tuple(int(v) for v in r) if ok else None


def count_pairs(splats, depths, width, height) -> int:
    lib = _load()
    s, d = _f32(splats).reshape(-1, 9), _f32(depths).reshape(-1)
    return int(lib.orc_count_pairs(_ptr(s), _ptr(d), s.shape[0], width, height))


def bin_splats(splats, depths, width, height):
    """Returns (keys u64[P], idx u32[P], ranges u32[T, 2])."""
    lib = _load()
    s, d = _f32(splats).reshape(-1, 9), _f32(depths).reshape(-1)
    p = count_pairs(s, d, width, height)
    tx, ty = tiles(width, height)
    keys = np.zeros(max(p, 1), dtype=np.uint64)
    idx = np.zeros(max(p, 1), dtype=np.uint32)
    ranges = np.zeros((tx * ty, 2), dtype=np.uint32)
    got = lib.orc_bin(_ptr(s), _ptr(d), s.shape[0], width, height, _ptr(keys), _ptr(idx),
                      _ptr(ranges), p)
    assert got == p
    return keys[:p], idx[:p], ranges


def radix_passes_4bit(num_tiles: int) -> int:
    return int(_load().orc_radix_passes_4bit(num_tiles))


def forward(splats, idx, ranges, width, height, *, f64=False, eps_alpha=0.0, sigma_ulps=8.0):
    """Tiled forward.  Returns dict(out [H*W,4], final_T, last, margin, counters)."""
    lib = _load()
    dt = np.float64 if f64 else np.float32
    s = np.ascontiguousarray(splats, dtype=dt).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    npx = width * height
    out = np.zeros((npx, 4), dtype=dt)
    final_t = np.zeros(npx, dtype=dt)
    last = np.zeros(npx, dtype=np.uint32)
    margin = np.zeros(npx, dtype=np.float32)
    cnt = np.zeros(3, dtype=np.int64)
    fn = lib.orc_forward_f64 if f64 else lib.orc_forward_f32
    fn(_ptr(s), _ptr(ix), _ptr(rg), width, height, _ptr(out), _ptr(final_t), _ptr(last),
       _ptr(margin), float(eps_alpha), float(sigma_ulps), _ptr(cnt))
    return {"out": out, "final_T": final_t, "last": last, "margin": margin,
            "counters": {"n_eval": int(cnt[0]), "n_exp": int(cnt[1]), "n_contrib": int(cnt[2])}}


def forward_untiled(splats, depths, width, height, *, sigma_skip=True, box=True):
    """Brute force over all splats per pixel.  box=False drops the 3-sigma box
    predicate (a diagnostic of the colour the box truncates)."""
    lib = _load()
    s, d = _f32(splats).reshape(-1, 9), _f32(depths).reshape(-1)
    npx = width * height
    out = np.zeros((npx, 4), dtype=np.float32)
    final_t = np.zeros(npx, dtype=np.float32)
    last = np.zeros(npx, dtype=np.uint32)
    if not box:
        fn = lib.orc_forward_untiled_nobox_f32
    else:
        fn = lib.orc_forward_untiled_f32 if sigma_skip else lib.orc_forward_untiled_noskip_f32
    fn(_ptr(s), _ptr(d), s.shape[0], width, height, _ptr(out), _ptr(final_t), _ptr(last))
    return {"out": out, "final_T": final_t, "last": last}


def backward(splats, idx, ranges, width, height, dl_dout, *, f64=False, eps_alpha=0.0,
             sigma_ulps=8.0):
    """Returns dict(grad float64 [N,9], gabs float64 [N,9] (sum of |per-pixel term|),
    knife bool [N], counters)."""
    lib = _load()
    dt = np.float64 if f64 else np.float32
    s = np.ascontiguousarray(splats, dtype=dt).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    g = np.ascontiguousarray(dl_dout, dtype=dt).reshape(-1, 4)
    n = s.shape[0]
    grad = np.zeros((n, 9), dtype=np.float64)
    gabs = np.zeros((n, 9), dtype=np.float64)
    knife = np.zeros(n, dtype=np.uint8)
    cnt = np.zeros(3, dtype=np.int64)
    fn = lib.orc_backward_f64 if f64 else lib.orc_backward_f32
    fn(_ptr(s), n, _ptr(ix), _ptr(rg), width, height, _ptr(g), _ptr(grad), _ptr(gabs), _ptr(knife),
       float(eps_alpha), float(sigma_ulps), _ptr(cnt))
    return {"grad": grad, "gabs": gabs, "knife": knife.astype(bool),
            "counters": {"n_eval": int(cnt[0]), "n_exp": int(cnt[1]), "n_contrib": int(cnt[2])}}


# --- forced replays ---------------------------------------------------------

# Decisions a forced replay may take the other way (oracle.h): alpha against
# 1/255, next_T against 1e-4 (the stop), raw against 0.999 (the clamp).
DEC_ALPHA, DEC_STOP, DEC_CLAMP = 1, 2, 4
FLIP_DTYPE = np.dtype([("pixel", "<i8"), ("pos", "<u4"), ("type", "<u4")])
DECISION_DTYPE = np.dtype([("pos", "<u4"), ("type", "<u4"), ("splat", "<u4"), ("margin", "<f4")])


def flip_table(entries=()):
    """A flip table sorted by (pixel, pos) from (pixel, pos, type) triples;
    entries of the same (pixel, pos) are merged."""
    merged = {}
    for pixel, pos, typ in entries:
        key = (int(pixel), int(pos))
        merged[key] = merged.get(key, 0) | int(typ)
    t = np.zeros(len(merged), dtype=FLIP_DTYPE)
    for k, ((pixel, pos), typ) in enumerate(sorted(merged.items())):
        t[k] = (pixel, pos, typ)
    return t


def _flips(table):
    t = np.ascontiguousarray(table if table is not None else np.zeros(0, FLIP_DTYPE), dtype=FLIP_DTYPE)
    return t, len(t)


def forward_forced(splats, idx, ranges, width, height, flips, *, eps_alpha, sigma_ulps=0.0):
    """The f32 forward with the decisions of `flips` taken the other way.
    Returns dict(out, final_T, last, refused)."""
    lib = _load()
    s = _f32(splats).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    t, nt = _flips(flips)
    npx = width * height
    out = np.zeros((npx, 4), dtype=np.float32)
    final_t = np.zeros(npx, dtype=np.float32)
    last = np.zeros(npx, dtype=np.uint32)
    refused = np.zeros(1, dtype=np.int64)
    lib.orc_forward_forced_f32(_ptr(s), _ptr(ix), _ptr(rg), width, height, _ptr(t), nt, _ptr(out),
                               _ptr(final_t), _ptr(last), float(eps_alpha), float(sigma_ulps), _ptr(refused))
    return {"out": out, "final_T": final_t, "last": last, "refused": int(refused[0])}


def pixel_forced(splats, idx, ranges, width, height, px, py, flips, *, eps_alpha, sigma_ulps=0.0,
                 max_decisions=256):
    """One pixel's forced forward: (out5 = rgb, w, final_T; last; the decisions
    within their uncertainty along it; refused flips)."""
    lib = _load()
    s = _f32(splats).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    t, nt = _flips(flips)
    out5 = np.zeros(5, dtype=np.float32)
    last = np.zeros(1, dtype=np.uint32)
    dec = np.zeros(max_decisions, dtype=DECISION_DTYPE)
    ndec = np.zeros(1, dtype=np.int32)
    refused = np.zeros(1, dtype=np.int64)
    lib.orc_pixel_forced_f32(_ptr(s), _ptr(ix), _ptr(rg), width, height, int(px), int(py), _ptr(t), nt,
                             float(eps_alpha), float(sigma_ulps), _ptr(out5), _ptr(last), _ptr(dec),
                             max_decisions, _ptr(ndec), _ptr(refused))
    return out5, int(last[0]), dec[:ndec[0]].copy(), int(refused[0])


def backward_forced(splats, idx, ranges, width, height, dl_dout, flips, *, eps_alpha, sigma_ulps=0.0):
    """The f32 backward (double sums) with the decisions of `flips` taken the
    other way.  Returns dict(grad [N,9], gabs [N,9], refused)."""
    lib = _load()
    s = _f32(splats).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    g = _f32(dl_dout).reshape(-1, 4)
    t, nt = _flips(flips)
    n = s.shape[0]
    grad = np.zeros((n, 9), dtype=np.float64)
    gabs = np.zeros((n, 9), dtype=np.float64)
    refused = np.zeros(1, dtype=np.int64)
    lib.orc_backward_forced_f32(_ptr(s), n, _ptr(ix), _ptr(rg), width, height, _ptr(g), _ptr(t), nt,
                                _ptr(grad), _ptr(gabs), float(eps_alpha), float(sigma_ulps), _ptr(refused))
    return {"grad": grad, "gabs": gabs, "refused": int(refused[0])}


def backward_targets(splats, idx, ranges, width, height, dl_dout, flips, targets, *, eps_alpha,
                     sigma_ulps=0.0):
    """The forced backward's gradients of the splats `targets` only.
    Returns (grad [k,9], gabs [k,9], refused)."""
    lib = _load()
    s = _f32(splats).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    g = _f32(dl_dout).reshape(-1, 4)
    t, nt = _flips(flips)
    tg = np.ascontiguousarray(targets, dtype=np.uint32).reshape(-1)
    grad = np.zeros((len(tg), 9), dtype=np.float64)
    gabs = np.zeros((len(tg), 9), dtype=np.float64)
    refused = np.zeros(1, dtype=np.int64)
    lib.orc_backward_targets_f32(_ptr(s), s.shape[0], _ptr(ix), _ptr(rg), width, height, _ptr(g), _ptr(t), nt,
                                 _ptr(tg), len(tg), _ptr(grad), _ptr(gabs), float(eps_alpha), float(sigma_ulps),
                                 _ptr(refused))
    return grad, gabs, int(refused[0])


def pixel_backward_forced(splats, idx, ranges, width, height, dl_dout, px, py, flips, target, *, eps_alpha,
                          sigma_ulps=0.0):
    """Splat `target`'s gradient terms at pixel (px, py) under the flips:
    (terms float64 [9], refused)."""
    lib = _load()
    s = _f32(splats).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    g = _f32(dl_dout).reshape(-1, 4)
    t, nt = _flips(flips)
    out = np.zeros(9, dtype=np.float64)
    refused = np.zeros(1, dtype=np.int64)
    lib.orc_pixel_backward_forced_f32(_ptr(s), _ptr(ix), _ptr(rg), width, height, _ptr(g), int(px), int(py),
                                      _ptr(t), nt, int(target), _ptr(out), float(eps_alpha), float(sigma_ulps),
                                      _ptr(refused))
    return out, int(refused[0])


def splat_decisions(splats, idx, ranges, width, height, flips, target, *, eps_alpha, sigma_ulps=0.0,
                    max_decisions=4096):
    """Splat `target`'s own decisions within their uncertainty at every pixel it
    is evaluated at: (flip-table entries, margins)."""
    lib = _load()
    s = _f32(splats).reshape(-1, 9)
    ix = np.ascontiguousarray(idx, dtype=np.uint32)
    rg = np.ascontiguousarray(ranges, dtype=np.uint32)
    t, nt = _flips(flips)
    out = np.zeros(max_decisions, dtype=FLIP_DTYPE)
    margins = np.zeros(max_decisions, dtype=np.float32)
    count = np.zeros(1, dtype=np.int32)
    lib.orc_splat_decisions_f32(_ptr(s), s.shape[0], _ptr(ix), _ptr(rg), width, height, _ptr(t), nt,
                                int(target), float(eps_alpha), float(sigma_ulps), _ptr(out), _ptr(margins),
                                max_decisions, _ptr(count))
    return out[:count[0]].copy(), margins[:count[0]].copy()


# --- projection (project.c) -------------------------------------------------

GAUSSIAN_FIELDS = 14   # mean xyz, log_scale xyz, quat wxyz, logit_opacity, rgb
CAMERA_FIELDS = 18     # W row-major (9), t (3), fx, fy, cx, cy, z_near, eps


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def project_forward(gaussians, camera):
    """Returns (splats float64 [n,9], depths float64 [n], visible bool [n])."""
    lib = _load()
    g = _f64(gaussians).reshape(-1, GAUSSIAN_FIELDS)
    cam = _f64(camera).reshape(CAMERA_FIELDS)
    n = g.shape[0]
    splats = np.zeros((n, 9), dtype=np.float64)
    depths = np.zeros(n, dtype=np.float64)
    vis = np.zeros(n, dtype=np.uint8)
    lib.orc_project_forward(_ptr(g), n, _ptr(cam), _ptr(splats), _ptr(depths), _ptr(vis))
    return splats, depths, vis.astype(bool)


def project_backward(gaussians, camera, dl_dsplat, with_abs=False):
    """Returns dL/dgaussians float64 [n,14] for dL/dsplat [n,9]; with_abs: also
    the sum of |terms| of each output's last sum, [n,14]."""
    lib = _load()
    g = _f64(gaussians).reshape(-1, GAUSSIAN_FIELDS)
    cam = _f64(camera).reshape(CAMERA_FIELDS)
    d = _f64(dl_dsplat).reshape(-1, 9)
    out = np.zeros_like(g)
    gabs = np.zeros_like(g) if with_abs else None
    lib.orc_project_backward(_ptr(g), g.shape[0], _ptr(cam), _ptr(d), _ptr(out),
                             _ptr(gabs) if with_abs else None)
    return (out, gabs) if with_abs else out

