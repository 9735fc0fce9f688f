"""GB300-native tile-binned 2-D Gaussian splat rasterizer.

The compute path is libgsr.so (hand-written sm_103a CUDA kernels behind the C
ABI in include/gsr.h); this package is its thin Python binding:

    ctx = Context(0)
    bins = bin_splats(ctx, splats, depths, width, height)
    out_rgbw, final_T, last = rasterize_forward(ctx, splats, bins)
    grad = rasterize_backward(ctx, splats, bins, dl_dout, final_T, last)

and on either side the projection of 3-D Gaussians and its backward:

    splats, depths = project_forward(ctx, gaussians, camera)
    dl_dgaussians = project_backward(ctx, gaussians, camera, grad)
"""
from ._abi import (LIB_PATH, Bins, Context, GsrError, bin_splats, peak_kernel, project_backward,
                   project_forward, rasterize_backward, rasterize_forward)

__all__ = ["LIB_PATH", "Bins", "Context", "GsrError", "bin_splats", "rasterize_forward",
           "rasterize_backward", "project_forward", "project_backward", "peak_kernel"]
