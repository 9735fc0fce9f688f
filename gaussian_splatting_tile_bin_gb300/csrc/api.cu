// api.cu -- the extern "C" surface of libgsr.so: argument checks, the device
// guard, error reporting and the context / arena lifetime.  The operations
// themselves live in bin.cu and raster.cu.
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <new>
#include <string>

#include "internal.cuh"

namespace gsr {

int fail(gsr_ctx *ctx, int code, const std::string &msg)
{
    if (ctx) ctx->err = msg;
    return code;
}

int cuda_check(gsr_ctx *ctx, cudaError_t e, const char *what)
{
    if (e == cudaSuccess) return GSR_OK;
    return fail(ctx, GSR_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

namespace {

// Makes the context's device current for the lifetime of the guard.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            cudaGetLastError();
            prev = -1;
        }
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// An NVTX range named after the entry point, for profilers' timelines (a no-op
// unless a tool is attached).
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
};

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_bins(gsr_ctx *ctx, const gsr_bins *bins, int32_t n)
{
    if (!bins) return fail(ctx, GSR_ERR_INVALID_ARG, "bins is NULL");
    if (bins->n != n) return fail(ctx, GSR_ERR_INVALID_ARG, "n differs from the n the bins were built from");
    if (bins->width < 1 || bins->height < 1 || bins->width > GSR_MAX_IMAGE_SIDE ||
        bins->height > GSR_MAX_IMAGE_SIDE)
        return fail(ctx, GSR_ERR_INVALID_ARG, "bins carry an invalid image size");
    if (bins->tiles_x != (bins->width + GSR_TILE - 1) / GSR_TILE ||
        bins->tiles_y != (bins->height + GSR_TILE - 1) / GSR_TILE)
        return fail(ctx, GSR_ERR_INVALID_ARG, "bins carry an inconsistent tile grid");
    if (!bins->tile_ranges || (n > 0 && bins->num_pairs > 0 && !bins->sorted_idx))
        return fail(ctx, GSR_ERR_INVALID_ARG, "bins hold NULL arrays");
    return GSR_OK;
}

}  // namespace
}  // namespace gsr

using namespace gsr;

extern "C" {

int gsr_create(gsr_ctx **out, int device)
{
    if (!out) return GSR_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
        cudaGetLastError();
        return GSR_ERR_CUDA;
    }
    if (device < 0 || device >= count) return GSR_ERR_INVALID_ARG;
    // Grid sizes of the grid-stride kernels are multiples of the SM count.
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return GSR_ERR_CUDA;
    }
    gsr_ctx *ctx = new (std::nothrow) gsr_ctx();
    if (!ctx) return GSR_ERR_OOM;
    ctx->device = device;
    ctx->num_sms = sms;
    *out = ctx;
    return GSR_OK;
}

void gsr_destroy(gsr_ctx *ctx)
{
    if (!ctx) return;
    {
        DeviceGuard g(ctx->device);
        for (int b = 0; b < 3; ++b) {
            cudaFree(ctx->pairs.k[b]);
            cudaFree(ctx->pairs.v[b]);
        }
        cudaFree(ctx->rects);
        for (int b = 0; b < 3; ++b) {
            cudaFree(ctx->depth.k[b]);
            cudaFree(ctx->depth.v[b]);
        }
        cudaFree(ctx->blk_sums);
        cudaFree(ctx->ranges);
        cudaFree(ctx->radix_counts);
        cudaFree(ctx->radix_totals);
        cudaFree(ctx->scalars);
        cudaFree(ctx->grad_acc);
        cudaFree(ctx->bwd_tile_cost);
        cudaFree(ctx->det_escale);
        cudaFree(ctx->bnd);
        cudaFree(ctx->bwd_items);
        cudaFree(ctx->fwd_items);
        if (ctx->host_total) cudaFreeHost(ctx->host_total);
    }
    delete ctx;
}

const char *gsr_last_error(const gsr_ctx *ctx) { return ctx ? ctx->err.c_str() : "NULL context"; }

int gsr_set_option(gsr_ctx *ctx, int option, int value)
{
    if (!ctx) return GSR_ERR_INVALID_ARG;
    if (value != 0 && value != 1) return fail(ctx, GSR_ERR_INVALID_ARG, "option value must be 0 or 1");
    switch (option) {
    case GSR_OPT_BWD_WARP_SKIP: ctx->opt_warp_skip = value; return GSR_OK;
    case GSR_OPT_BWD_LAST_CONTRIB: ctx->opt_last_contrib = value; return GSR_OK;
    case GSR_OPT_WARP_CULL: ctx->opt_warp_cull = value; return GSR_OK;
    case GSR_OPT_PDL: ctx->opt_pdl = value; return GSR_OK;
    case GSR_OPT_FAIL_NEXT_ALLOC: ctx->fail_next_alloc = value; return GSR_OK;
    case GSR_OPT_DETERMINISTIC: ctx->opt_deterministic = value; return GSR_OK;
    case GSR_OPT_BWD_PER_SPLAT: ctx->opt_bwd_per_splat = value; return GSR_OK;
    case GSR_OPT_SPLIT: ctx->opt_split = value; return GSR_OK;
    case GSR_OPT_SPLIT_FORWARD: ctx->opt_split_forward = value; return GSR_OK;
    default: return fail(ctx, GSR_ERR_INVALID_ARG, "unknown option " + std::to_string(option));
    }
}

uint64_t gsr_launch_count(const gsr_ctx *ctx) { return ctx ? ctx->launches : 0; }

int gsr_bin_splats(gsr_ctx *ctx, const gsr_splat2d *splats, const float *depths, int32_t n,
                   int32_t width, int32_t height, void *stream, gsr_bins *out)
{
    gsr::Range range("gsr_bin_splats");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    if (!out) return fail(ctx, GSR_ERR_INVALID_ARG, "out is NULL");
    if (n < 0 || n > GSR_MAX_SPLATS) return fail(ctx, GSR_ERR_INVALID_ARG, "n out of range");
    if (width < 1 || height < 1 || width > GSR_MAX_IMAGE_SIDE || height > GSR_MAX_IMAGE_SIDE)
        return fail(ctx, GSR_ERR_INVALID_ARG, "width/height out of range");
    if (n > 0 && (!splats || !depths)) return fail(ctx, GSR_ERR_INVALID_ARG, "splats/depths is NULL");
    if (!aligned(splats, 4) || !aligned(depths, 4))
        return fail(ctx, GSR_ERR_INVALID_ARG, "splats/depths must be 4-byte aligned");
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    return gsr::bin_splats(ctx, reinterpret_cast<const float *>(splats), depths, n, width, height,
                           (cudaStream_t)stream, out);
}

int gsr_rasterize_forward(gsr_ctx *ctx, const gsr_splat2d *splats, int32_t n, const gsr_bins *bins,
                          float *out_rgbw, float *final_T, uint32_t *last_contrib, void *stream)
{
    gsr::Range range("gsr_rasterize_forward");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    int rc = check_bins(ctx, bins, n);
    if (rc) return rc;
    if (!out_rgbw || !final_T || !last_contrib)
        return fail(ctx, GSR_ERR_INVALID_ARG, "an output pointer is NULL");
    if (n > 0 && bins->num_pairs > 0 && !splats) return fail(ctx, GSR_ERR_INVALID_ARG, "splats is NULL");
    if (!aligned(out_rgbw, 16) || !aligned(final_T, 4) || !aligned(last_contrib, 4) ||
        !aligned(splats, 4))
        return fail(ctx, GSR_ERR_INVALID_ARG, "misaligned buffer (out_rgbw needs 16 bytes)");
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    return gsr::rasterize_forward(ctx, reinterpret_cast<const float *>(splats), bins, out_rgbw, final_T,
                                  last_contrib, (cudaStream_t)stream);
}

int gsr_rasterize_backward(gsr_ctx *ctx, const gsr_splat2d *splats, int32_t n, const gsr_bins *bins,
                           const float *dl_dout, const float *final_T, const uint32_t *last_contrib,
                           float *grad, void *stream)
{
    gsr::Range range("gsr_rasterize_backward");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    int rc = check_bins(ctx, bins, n);
    if (rc) return rc;
    if (!dl_dout || !final_T || !last_contrib || (n > 0 && !grad))
        return fail(ctx, GSR_ERR_INVALID_ARG, "an input/output pointer is NULL");
    if (n > 0 && bins->num_pairs > 0 && !splats) return fail(ctx, GSR_ERR_INVALID_ARG, "splats is NULL");
    if (!aligned(dl_dout, 16) || !aligned(final_T, 4) || !aligned(last_contrib, 4) ||
        !aligned(grad, 4) || !aligned(splats, 4))
        return fail(ctx, GSR_ERR_INVALID_ARG, "misaligned buffer (dl_dout needs 16 bytes)");
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    if (n == 0) return GSR_OK;
    return gsr::rasterize_backward(ctx, reinterpret_cast<const float *>(splats), n, bins, dl_dout,
                                   final_T, last_contrib, grad, (cudaStream_t)stream);
}

int gsr_rasterize_backward_noalloc(gsr_ctx *ctx, const gsr_splat2d *splats, int32_t n,
                                   const gsr_bins *bins, const float *dl_dout, const float *final_T,
                                   const uint32_t *last_contrib, float *grad, void *stream)
{
    gsr::Range range("gsr_rasterize_backward_noalloc");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    if (n < 0 || n > GSR_NOALLOC_MAX_SPLATS)
        return fail(ctx, GSR_ERR_INVALID_ARG,
                    "n = " + std::to_string(n) + " is outside [0, GSR_NOALLOC_MAX_SPLATS = " +
                        std::to_string(GSR_NOALLOC_MAX_SPLATS) + "]");
    int rc = check_bins(ctx, bins, n);
    if (rc) return rc;
    if (!dl_dout || !final_T || !last_contrib || (n > 0 && !grad))
        return fail(ctx, GSR_ERR_INVALID_ARG, "an input/output pointer is NULL");
    if (n > 0 && bins->num_pairs > 0 && !splats) return fail(ctx, GSR_ERR_INVALID_ARG, "splats is NULL");
    if (!aligned(dl_dout, 16) || !aligned(final_T, 4) || !aligned(last_contrib, 4) ||
        !aligned(grad, 4) || !aligned(splats, 4))
        return fail(ctx, GSR_ERR_INVALID_ARG, "misaligned buffer (dl_dout needs 16 bytes)");
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    if (n == 0) return GSR_OK;
    return gsr::rasterize_backward_noalloc(ctx, reinterpret_cast<const float *>(splats), n, bins,
                                           dl_dout, final_T, last_contrib, grad,
                                           (cudaStream_t)stream);
}

int gsr_get_bin_stats(gsr_ctx *ctx, gsr_bin_stats *out)
{
    if (!ctx || !out) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    DeviceGuard g(ctx->device);
    *out = gsr_bin_stats{};
    out->capacity = ctx->cap_pairs;
    uint32_t status = GSR_OK;
    int rc = gsr::bin_result(ctx, &out->num_pairs, &status, &out->emitting);
    if (rc) return rc;
    int tile_bits = 0, tile_digits = 0;
    rc = gsr::bin_pass_masks(ctx, &out->depth_pass_mask, &out->tile_pass_mask, &tile_bits, &tile_digits);
    if (rc) return rc;
    out->tile_digit_bits = tile_bits;
    out->tile_digits = tile_digits;
    out->radix_passes = __builtin_popcount(out->depth_pass_mask) + __builtin_popcount(out->tile_pass_mask);
    return GSR_OK;
}

int gsr_reserve_pairs(gsr_ctx *ctx, uint64_t max_pairs)
{
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    if (max_pairs > (uint64_t)GSR_MAX_PAIRS)
        return fail(ctx, GSR_ERR_INVALID_ARG, "max_pairs exceeds GSR_MAX_PAIRS");
    ctx->reserved_pairs = max_pairs;
    return GSR_OK;
}

int gsr_num_pairs(gsr_ctx *ctx, uint32_t *out)
{
    if (!ctx || !out) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    uint32_t status = GSR_OK;
    int rc = gsr::bin_result(ctx, out, &status, nullptr);
    if (rc) return rc;
    if (status != GSR_OK)
        return fail(ctx, GSR_ERR_TOO_MANY_PAIRS,
                    "the last binning needed " + std::to_string(*out) + " tile pairs, more than the arena's " +
                        std::to_string(ctx->cap_pairs) + ": its bins are empty");
    return GSR_OK;
}

int gsr_exp_neg(gsr_ctx *ctx, const float *s, float *out, int32_t n, void *stream)
{
    gsr::Range range("gsr_exp_neg");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    if (n < 0) return fail(ctx, GSR_ERR_INVALID_ARG, "n < 0");
    if (n > 0 && (!s || !out)) return fail(ctx, GSR_ERR_INVALID_ARG, "s/out is NULL");
    if (!aligned(s, 4) || !aligned(out, 4)) return fail(ctx, GSR_ERR_INVALID_ARG, "s/out must be 4-byte aligned");
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    if (n == 0) return GSR_OK;
    return gsr::exp_neg_eval(ctx, s, out, n, (cudaStream_t)stream);
}

int gsr_peak_kernel(gsr_ctx *ctx, int kind, int32_t iters, float *sink, uint64_t *lane_ops, void *stream)
{
    gsr::Range range("gsr_peak_kernel");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    if (kind != GSR_PEAK_FFMA && kind != GSR_PEAK_EX2) return fail(ctx, GSR_ERR_INVALID_ARG, "unknown peak kind");
    if (iters < 1 || iters > (1 << 24)) return fail(ctx, GSR_ERR_INVALID_ARG, "iters outside [1, 2^24]");
    if (!sink || !lane_ops) return fail(ctx, GSR_ERR_INVALID_ARG, "sink/lane_ops is NULL");
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    return gsr::peak_kernel(ctx, kind, iters, sink, lane_ops, (cudaStream_t)stream);
}

}  // extern "C"

namespace {

int check_projection(gsr_ctx *ctx, const void *gauss, int32_t n, const gsr_camera *cam, const void *a,
                     const void *b)
{
    if (!cam) return fail(ctx, GSR_ERR_INVALID_ARG, "camera is NULL");
    if (n < 0 || n > GSR_MAX_SPLATS) return fail(ctx, GSR_ERR_INVALID_ARG, "n out of range");
    if (n > 0 && (!gauss || !a || !b)) return fail(ctx, GSR_ERR_INVALID_ARG, "an array is NULL");
    if (!aligned(gauss, 4) || !aligned(a, 4) || !aligned(b, 4))
        return fail(ctx, GSR_ERR_INVALID_ARG, "arrays must be 4-byte aligned");
    const float *f = reinterpret_cast<const float *>(cam);
    for (size_t k = 0; k < sizeof(gsr_camera) / sizeof(float); ++k)
        if (!std::isfinite(f[k])) return fail(ctx, GSR_ERR_INVALID_ARG, "camera field not finite");
    if (!(cam->z_near > 0.0f)) return fail(ctx, GSR_ERR_INVALID_ARG, "camera z_near must be > 0");
    if (!(cam->eps >= 0.0f)) return fail(ctx, GSR_ERR_INVALID_ARG, "camera eps must be >= 0");
    return GSR_OK;
}

}  // namespace

extern "C" {

int gsr_project_forward(gsr_ctx *ctx, const gsr_gaussian3d *gauss, int32_t n, const gsr_camera *camera,
                        gsr_splat2d *splats, float *depths, void *stream)
{
    gsr::Range range("gsr_project_forward");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    if (int rc = check_projection(ctx, gauss, n, camera, splats, depths)) return rc;
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    if (n == 0) return GSR_OK;
    return gsr::project_forward(ctx, reinterpret_cast<const float *>(gauss), n, *camera,
                                reinterpret_cast<float *>(splats), depths, (cudaStream_t)stream);
}

int gsr_project_backward(gsr_ctx *ctx, const gsr_gaussian3d *gauss, int32_t n, const gsr_camera *camera,
                         const float *dl_dsplat, float *dl_dgauss, void *stream)
{
    gsr::Range range("gsr_project_backward");
    if (!ctx) return GSR_ERR_INVALID_ARG;
    ctx->err.clear();
    if (int rc = check_projection(ctx, gauss, n, camera, dl_dsplat, dl_dgauss)) return rc;
    DeviceGuard g(ctx->device);
    if (!g.ok) return fail(ctx, GSR_ERR_CUDA, "cannot select the context's device");
    if (n == 0) return GSR_OK;
    return gsr::project_backward(ctx, reinterpret_cast<const float *>(gauss), n, *camera, dl_dsplat, dl_dgauss,
                                 (cudaStream_t)stream);
}

}  // extern "C"

static_assert(sizeof(gsr_splat2d) == 36, "Splat2D is 9 floats");
static_assert(sizeof(gsr_gaussian3d) == GSR_GAUSSIAN_FLOATS * 4, "a Gaussian is 14 floats");
static_assert(sizeof(gsr_camera) == 18 * 4, "a camera is 18 floats");
