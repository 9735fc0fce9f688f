"""ctypes binding of libgsr.so: argument checks and marshalling only.

Every step of binning, forward and backward runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  When libgsr.so is
missing, importing this module raises: there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# GSR_LIBRARY selects another build of the same library (A/B of build flags).
LIB_PATH = os.environ.get("GSR_LIBRARY") or os.path.join(_PKG, "lib", "libgsr.so")

GSR_OK, GSR_ERR_INVALID_ARG, GSR_ERR_CUDA, GSR_ERR_OOM, GSR_ERR_TOO_MANY_PAIRS = range(5)
GSR_PAIRS_ON_DEVICE = 0xFFFFFFFF
OPTIONS = {"bwd_warp_skip": 1, "bwd_last_contrib": 2, "warp_cull": 3, "pdl": 4, "fail_next_alloc": 5,
           "deterministic": 6, "bwd_per_splat": 7, "split": 8, "split_forward": 9}


class GsrError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"gsr error {code}: {msg}")
        self.code = code


class _Bins(ctypes.Structure):
    _fields_ = [("keys", ctypes.c_void_p), ("sorted_idx", ctypes.c_void_p),
                ("tile_ranges", ctypes.c_void_p), ("tile_order", ctypes.c_void_p),
                ("num_pairs_dev", ctypes.c_void_p), ("num_pairs", ctypes.c_uint32),
                ("n", ctypes.c_int32), ("width", ctypes.c_int32), ("height", ctypes.c_int32),
                ("tiles_x", ctypes.c_int32), ("tiles_y", ctypes.c_int32)]


GAUSSIAN_FIELDS = 14   # mean xyz, log_scale xyz, quat wxyz, logit_opacity, rgb
CAMERA_FIELDS = 18     # W row-major (9), t (3), fx, fy, cx, cy, z_near, eps


class _Camera(ctypes.Structure):
    _fields_ = [("v", ctypes.c_float * CAMERA_FIELDS)]


class _BinStats(ctypes.Structure):
    _fields_ = [("num_pairs", ctypes.c_uint32), ("emitting", ctypes.c_uint32),
                ("radix_passes", ctypes.c_int32), ("depth_pass_mask", ctypes.c_uint32),
                ("tile_pass_mask", ctypes.c_uint32), ("tile_digit_bits", ctypes.c_int32),
                ("tile_digits", ctypes.c_int32), ("capacity", ctypes.c_uint64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.gsr_create.argtypes = [ctypes.POINTER(P), ctypes.c_int]
    lib.gsr_create.restype = ctypes.c_int
    lib.gsr_destroy.argtypes = [P]
    lib.gsr_destroy.restype = None
    lib.gsr_last_error.argtypes = [P]
    lib.gsr_last_error.restype = ctypes.c_char_p
    lib.gsr_set_option.argtypes = [P, ctypes.c_int, ctypes.c_int]
    lib.gsr_set_option.restype = ctypes.c_int
    lib.gsr_launch_count.argtypes = [P]
    lib.gsr_launch_count.restype = ctypes.c_uint64
    lib.gsr_bin_splats.argtypes = [P, P, P, i32, i32, i32, P, ctypes.POINTER(_Bins)]
    lib.gsr_bin_splats.restype = ctypes.c_int
    lib.gsr_rasterize_forward.argtypes = [P, P, i32, ctypes.POINTER(_Bins), P, P, P, P]
    lib.gsr_rasterize_forward.restype = ctypes.c_int
    lib.gsr_rasterize_backward.argtypes = [P, P, i32, ctypes.POINTER(_Bins), P, P, P, P, P]
    lib.gsr_rasterize_backward.restype = ctypes.c_int
    lib.gsr_reserve_pairs.argtypes = [P, ctypes.c_uint64]
    lib.gsr_reserve_pairs.restype = ctypes.c_int
    lib.gsr_num_pairs.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.gsr_num_pairs.restype = ctypes.c_int
    lib.gsr_get_bin_stats.argtypes = [P, ctypes.POINTER(_BinStats)]
    lib.gsr_get_bin_stats.restype = ctypes.c_int
    lib.gsr_project_forward.argtypes = [P, P, i32, ctypes.POINTER(_Camera), P, P, P]
    lib.gsr_project_forward.restype = ctypes.c_int
    lib.gsr_project_backward.argtypes = [P, P, i32, ctypes.POINTER(_Camera), P, P, P]
    lib.gsr_project_backward.restype = ctypes.c_int
    lib.gsr_exp_neg.argtypes = [P, P, P, i32, P]
    lib.gsr_exp_neg.restype = ctypes.c_int
    lib.gsr_peak_kernel.argtypes = [P, ctypes.c_int, i32, P, ctypes.POINTER(ctypes.c_uint64), P]
    lib.gsr_peak_kernel.restype = ctypes.c_int
    return lib


lib = _load()


class _DeviceArray:
    """Minimal __cuda_array_interface__ holder for a view of arena memory."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"data": (int(ptr or 0), False), "shape": tuple(shape),
                                         "typestr": typestr, "version": 3, "strides": None}


class Context:
    """Owns a libgsr context (the grow-only binning arena) on one CUDA device."""

    def __init__(self, device: int = 0):
        h = ctypes.c_void_p()
        rc = lib.gsr_create(ctypes.byref(h), int(device))
        if rc != GSR_OK:
            raise GsrError(rc, "gsr_create failed")
        self._h = h
        self.device = int(device)
        # Bumped by every bin_splats: bins from an earlier call may point into
        # arena buffers that call freed or overwrote.
        self._bin_generation = 0

    def _check(self, rc):
        if rc != GSR_OK:
            raise GsrError(rc, lib.gsr_last_error(self._h).decode())

    def set_option(self, name: str, value: bool):
        """Sets a GSR_OPT_* switch by its name in OPTIONS (the header documents
        each): "split" (backward segments of crowded tiles, on by default),
        "split_forward" (the forward's chunks past a head, off by default),
        "deterministic", "bwd_per_splat", and the A/B switches."""
        self._check(lib.gsr_set_option(self._h, OPTIONS[name], int(bool(value))))

    def launch_count(self) -> int:
        return int(lib.gsr_launch_count(self._h))

    def reserve_pairs(self, max_pairs: int):
        """Sizes the arena for max_pairs tile pairs; later bin_splats calls
        read nothing back to the host (0: back to reading the count)."""
        self._check(lib.gsr_reserve_pairs(self._h, int(max_pairs)))

    def num_pairs(self) -> int:
        """The last binning's pair count (waits for it); GsrError with code
        GSR_ERR_TOO_MANY_PAIRS when it exceeded the reservation."""
        out = ctypes.c_uint32()
        self._check(lib.gsr_num_pairs(self._h, ctypes.byref(out)))
        return int(out.value)

    def bin_stats(self) -> dict:
        st = _BinStats()
        self._check(lib.gsr_get_bin_stats(self._h, ctypes.byref(st)))
        return {name: (int(getattr(st, name))) for name, _ in _BinStats._fields_}

    def close(self):
        if getattr(self, "_h", None):
            lib.gsr_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Bins:
    """Result of bin_splats: device views into the context's arena (valid until
    the next bin_splats on the same context, which may free or overwrite the
    buffers; later use raises ValueError)."""

    def __init__(self, ctx: Context, raw: _Bins, device, generation: int):
        self.ctx, self.raw, self._device, self.generation = ctx, raw, device, generation

    def _check_current(self):
        if getattr(self.ctx, "_h", None) is None:
            raise ValueError("the context these bins belong to is closed")
        if self.generation != self.ctx._bin_generation:
            raise ValueError("these bins were replaced by a later bin_splats on the same context")

    @property
    def num_pairs(self) -> int:
        """The pair count; for bins whose count stayed on the device this waits
        for the binning and reads it."""
        if int(self.raw.num_pairs) == GSR_PAIRS_ON_DEVICE:
            self._check_current()
            return self.ctx.num_pairs()
        return int(self.raw.num_pairs)

    @property
    def tiles(self):
        return int(self.raw.tiles_x), int(self.raw.tiles_y)

    def _view(self, ptr, shape, typestr):
        self._check_current()
        if shape[0] == 0:
            return torch.empty(shape, dtype={"<i8": torch.int64, "<i4": torch.int32}[typestr],
                               device=self._device)
        return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device=self._device)

    def keys(self) -> torch.Tensor:
        """Sorted keys as int64 (bit pattern of the uint64 keys)."""
        return self._view(self.raw.keys, (self.num_pairs,), "<i8")

    def sorted_idx(self) -> torch.Tensor:
        return self._view(self.raw.sorted_idx, (self.num_pairs,), "<i4")

    def tile_order(self) -> torch.Tensor:
        """Launch order of the tiles (longest lists first)."""
        tx, ty = self.tiles
        return self._view(self.raw.tile_order, (tx * ty,), "<i4")

    def tile_ranges(self) -> torch.Tensor:
        tx, ty = self.tiles
        return self._view(self.raw.tile_ranges, (tx * ty, 2), "<i4")


def exp_neg(ctx: Context, s: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """The raster kernels' exp(-s) on a device array (diagnostic)."""
    _need(s, "s", torch.float32)
    if out is None:
        out = torch.empty_like(s)
    _need(out, "out", torch.float32, tuple(s.shape))
    ctx._check(lib.gsr_exp_neg(ctx._h, ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                               int(s.numel()), _stream_ptr(stream, s.device)))
    return out


PEAK_KINDS = {"ffma": 0, "ex2": 1}


def peak_kernel(ctx: Context, kind: str, iters: int, sink: torch.Tensor, stream=None) -> int:
    """Enqueues one launch of the FP32 ("ffma") or SFU ("ex2") rate kernel;
    returns the number of lane operations it performs (time it with events)."""
    _need(sink, "sink", torch.float32)
    ops = ctypes.c_uint64()
    ctx._check(lib.gsr_peak_kernel(ctx._h, PEAK_KINDS[kind], int(iters), ctypes.c_void_p(sink.data_ptr()),
                                   ctypes.byref(ops), _stream_ptr(stream, sink.device)))
    return int(ops.value)


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def bin_splats(ctx: Context, splats: torch.Tensor, depths: torch.Tensor, width: int, height: int,
               stream=None) -> Bins:
    n = splats.shape[0] if splats.dim() == 2 else -1
    _need(splats, "splats", torch.float32, (n, 9))
    _need(depths, "depths", torch.float32, (n,))
    raw = _Bins()
    ctx._bin_generation += 1   # even a failed call may have regrown the arena
    ctx._check(lib.gsr_bin_splats(ctx._h, ctypes.c_void_p(splats.data_ptr()),
                                  ctypes.c_void_p(depths.data_ptr()), n, int(width), int(height),
                                  _stream_ptr(stream, splats.device), ctypes.byref(raw)))
    return Bins(ctx, raw, splats.device, ctx._bin_generation)


def rasterize_forward(ctx: Context, splats: torch.Tensor, bins: Bins, out_rgbw=None, final_T=None,
                      last_contrib=None, stream=None):
    """Returns (out_rgbw [H*W, 4] f32, final_T [H*W] f32, last_contrib [H*W] int32)."""
    bins._check_current()
    n = splats.shape[0]
    _need(splats, "splats", torch.float32, (n, 9))
    npx = int(bins.raw.width) * int(bins.raw.height)
    dev = splats.device
    if out_rgbw is None:
        out_rgbw = torch.empty((npx, 4), dtype=torch.float32, device=dev)
    if final_T is None:
        final_T = torch.empty((npx,), dtype=torch.float32, device=dev)
    if last_contrib is None:
        last_contrib = torch.empty((npx,), dtype=torch.int32, device=dev)
    _need(out_rgbw, "out_rgbw", torch.float32, (npx, 4))
    _need(final_T, "final_T", torch.float32, (npx,))
    _need(last_contrib, "last_contrib", torch.int32, (npx,))
    ctx._check(lib.gsr_rasterize_forward(
        ctx._h, ctypes.c_void_p(splats.data_ptr()), n, ctypes.byref(bins.raw),
        ctypes.c_void_p(out_rgbw.data_ptr()), ctypes.c_void_p(final_T.data_ptr()),
        ctypes.c_void_p(last_contrib.data_ptr()), _stream_ptr(stream, dev)))
    return out_rgbw, final_T, last_contrib


def rasterize_backward(ctx: Context, splats: torch.Tensor, bins: Bins, dl_dout: torch.Tensor,
                       final_T: torch.Tensor, last_contrib: torch.Tensor, grad=None, stream=None):
    """Returns grad [N, 9] f32 (d/d of each Splat2D field)."""
    bins._check_current()
    n = splats.shape[0]
    _need(splats, "splats", torch.float32, (n, 9))
    npx = int(bins.raw.width) * int(bins.raw.height)
    dev = splats.device
    if grad is None:
        grad = torch.empty((n, 9), dtype=torch.float32, device=dev)
    _need(dl_dout, "dl_dout", torch.float32, (npx, 4))
    _need(final_T, "final_T", torch.float32, (npx,))
    _need(last_contrib, "last_contrib", torch.int32, (npx,))
    _need(grad, "grad", torch.float32, (n, 9))
    ctx._check(lib.gsr_rasterize_backward(
        ctx._h, ctypes.c_void_p(splats.data_ptr()), n, ctypes.byref(bins.raw),
        ctypes.c_void_p(dl_dout.data_ptr()), ctypes.c_void_p(final_T.data_ptr()),
        ctypes.c_void_p(last_contrib.data_ptr()), ctypes.c_void_p(grad.data_ptr()),
        _stream_ptr(stream, dev)))
    return grad


def _camera(camera) -> _Camera:
    vals = [float(v) for v in (camera.tolist() if hasattr(camera, "tolist") else camera)]
    if len(vals) != CAMERA_FIELDS:
        raise ValueError(f"camera must hold {CAMERA_FIELDS} numbers (W row-major, t, fx, fy, cx, cy, "
                         "z_near, eps)")
    cam = _Camera()
    cam.v[:] = vals
    return cam


def project_forward(ctx: Context, gauss: torch.Tensor, camera, splats=None, depths=None, stream=None):
    """Projects 3-D Gaussians [n, 14] f32 through `camera` (18 numbers).
    Returns (splats [n, 9] f32, depths [n] f32)."""
    n = gauss.shape[0] if gauss.dim() == 2 else -1
    _need(gauss, "gauss", torch.float32, (n, GAUSSIAN_FIELDS))
    dev = gauss.device
    if splats is None:
        splats = torch.empty((n, 9), dtype=torch.float32, device=dev)
    if depths is None:
        depths = torch.empty((n,), dtype=torch.float32, device=dev)
    _need(splats, "splats", torch.float32, (n, 9))
    _need(depths, "depths", torch.float32, (n,))
    cam = _camera(camera)
    ctx._check(lib.gsr_project_forward(ctx._h, ctypes.c_void_p(gauss.data_ptr()), n, ctypes.byref(cam),
                                       ctypes.c_void_p(splats.data_ptr()), ctypes.c_void_p(depths.data_ptr()),
                                       _stream_ptr(stream, dev)))
    return splats, depths


def project_backward(ctx: Context, gauss: torch.Tensor, camera, dl_dsplat: torch.Tensor, dl_dgauss=None,
                     stream=None) -> torch.Tensor:
    """Returns dL/dgauss [n, 14] f32 for dL/dsplat [n, 9] f32."""
    n = gauss.shape[0] if gauss.dim() == 2 else -1
    _need(gauss, "gauss", torch.float32, (n, GAUSSIAN_FIELDS))
    _need(dl_dsplat, "dl_dsplat", torch.float32, (n, 9))
    dev = gauss.device
    if dl_dgauss is None:
        dl_dgauss = torch.empty((n, GAUSSIAN_FIELDS), dtype=torch.float32, device=dev)
    _need(dl_dgauss, "dl_dgauss", torch.float32, (n, GAUSSIAN_FIELDS))
    cam = _camera(camera)
    ctx._check(lib.gsr_project_backward(ctx._h, ctypes.c_void_p(gauss.data_ptr()), n, ctypes.byref(cam),
                                        ctypes.c_void_p(dl_dsplat.data_ptr()),
                                        ctypes.c_void_p(dl_dgauss.data_ptr()), _stream_ptr(stream, dev)))
    return dl_dgauss
