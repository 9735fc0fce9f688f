/*
 * gsr.h -- C ABI of libgsr.so, a tile-binned 2-D Gaussian splat rasterizer for
 * NVIDIA GB300 (sm_103a).
 *
 * Three entry points make one training iteration of the rasterizer:
 *   gsr_bin_splats          pairs each splat with the 16x16 tiles its 3-sigma box
 *                           touches and sorts the pairs by (tile, depth)
 *   gsr_rasterize_forward   front-to-back alpha compositing, one CTA per tile
 *   gsr_rasterize_backward  back-to-front replay giving d/d{mean, conic, rgb, color_a}
 *
 * The operations follow a 3D Gaussian Splatting trainer's findings pages:
 *   - "C0 resident arena + C1 pass skip" (p2-c0-resident-binning), section 2 table:
 *     pair keys (tile_id << 32) | depth_bits, a stable radix sort whose
 *     constant-digit passes are skipped, per-tile ranges, a grow-only arena;
 *   - "forward/adam audit" (p3-forward-adam-audit), sections (a), (b), (e), 3:
 *     one 256-thread group per 16x16 tile staging a batch of 256 Splat2D
 *     records, outputs rgb + final_T + last_contributor (24 B/pixel);
 *   - "A.9 f16 forward" (a-9-f16-forward-negative), implementation snippet:
 *     alpha = min(0.999, color_a exp(-sigma)), T <- T (1 - alpha), fp32 throughout;
 *   - "W1 warp sparse skip + exp-skip" (p2-w1-warp-sparse-skip), section 1: the
 *     sigma >= 5.55 skip, the all-lanes-idle warp skip before the reduction;
 *   - "M3 per-splat backward" (p3-per-splat-backward), section 1: 9 gradient
 *     components per splat, no background, no rgb clamp, alpha-clamp rule
 *     raw < 0.999.
 *
 * Conventions shared by every call
 *   - All array arguments are DEVICE pointers owned by the caller, except the
 *     arrays inside gsr_bins, which belong to the context's arena.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream).  gsr_bin_splats synchronises that stream once to
 *     read the pair count, unless the context has a reservation
 *     (gsr_reserve_pairs); the raster calls return without synchronising.
 *   - The calling thread's current CUDA device is switched to the context's
 *     device for the duration of a call and restored afterwards.
 *   - Every call returns GSR_OK or an error code; gsr_last_error() gives the text.
 *     No C++ exception crosses this interface.  A context is not thread-safe.
 *   - Pixel centres sit at integer coordinates (px, py); image sizes need not be
 *     multiples of 16 (pixels outside the image neither write nor contribute).
 */
#ifndef GSR_H
#define GSR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One splat after projection: 9 floats, 36 bytes, in this order
 * ("forward/adam audit", section 3, staging read: Splat2D = 9 float = 36 B).
 * The conic (a, b, c) is the inverse 2-D covariance: sigma(d) =
 * 1/2 (a dx^2 + c dy^2) + b dx dy.  color_a is expected in [0, 1]. */
typedef struct gsr_splat2d {
    float mean_x, mean_y;
    float conic_a, conic_b, conic_c;
    float color_r, color_g, color_b;
    float color_a;
} gsr_splat2d;

/* One 3-D Gaussian, the input of gsr_project_forward: 14 floats, 56 bytes.
 * quat is (w, x, y, z) and need not be normalised; the scales are exp(log_scale)
 * along the rotated axes; color_a = 1 / (1 + exp(-logit_opacity)). */
#define GSR_GAUSSIAN_FLOATS 14
typedef struct gsr_gaussian3d {
    float mean[3];
    float log_scale[3];
    float quat[4];
    float logit_opacity;
    float rgb[3];
} gsr_gaussian3d;

/* A pinhole camera: camera-space point p = W x + t (W row-major, usually a
 * rotation), pixel = (fx p.x / p.z + cx, fy p.y / p.z + cy).  Points with
 * p.z <= z_near are not projected.  eps is added to both diagonal entries of
 * every projected 2-D covariance (a low-pass dilation; 0 disables it). */
typedef struct gsr_camera {
    float W[9];
    float t[3];
    float fx, fy, cx, cy;
    float z_near;
    float eps;
} gsr_camera;

#define GSR_TILE 16
#define GSR_MAX_IMAGE_SIDE (1 << 19)   /* width and height limit */
#define GSR_MAX_SPLATS (1 << 28)       /* n limit */
#define GSR_MAX_PAIRS 0x7fffffffu      /* tile-pair limit (indices are uint32) */

enum {
    GSR_OK = 0,
    GSR_ERR_INVALID_ARG = 1,    /* null pointer, bad size or misaligned buffer */
    GSR_ERR_CUDA = 2,           /* a CUDA runtime call or launch failed */
    GSR_ERR_OOM = 3,            /* the arena could not grow */
    GSR_ERR_TOO_MANY_PAIRS = 4  /* more than GSR_MAX_PAIRS tile pairs */
};

/* Per-call variant switches (A/B and equivalence tests; defaults are 1). */
enum {
    GSR_OPT_BWD_WARP_SKIP = 1,   /* a warp skips the gradient arithmetic and reduction of a splat
                                    no lane composites */
    GSR_OPT_BWD_LAST_CONTRIB = 2, /* stop each warp at its largest last_contributor */
    GSR_OPT_WARP_CULL = 3,        /* forward and backward: a warp skips splats whose alpha >= 1/255
                                     ellipse misses its 8x4 pixel block (same results) */
    GSR_OPT_PDL = 4,              /* launch kernels with programmatic dependent launch: a kernel may
                                     begin launching while the one before it in the stream drains,
                                     and waits for it before touching memory (same results) */
    GSR_OPT_FAIL_NEXT_ALLOC = 5,  /* test hook (default 0): the context's next device allocation
                                     fails as if the GPU were out of memory; the call returns
                                     GSR_ERR_OOM and later calls allocate normally */
    GSR_OPT_DETERMINISTIC = 6,    /* default 0.  1: gsr_rasterize_backward accumulates in 64-bit fixed
                                     point (exponents chosen per splat from bounds on its terms), so
                                     its gradients are the same bits on every run, whatever order the
                                     warps add in ("M3 per-splat backward", sections 2 and 4: run-to-run
                                     self-noise).  A non-finite dL/dout makes every gradient NaN.  Not
                                     available to gsr_rasterize_backward_noalloc (GSR_ERR_INVALID_ARG). */
    GSR_OPT_BWD_PER_SPLAT = 7,    /* default 0.  1: the backward runs the transposed loop nest ("M3
                                     per-splat backward", section 1): one warp per tile, one lane per
                                     splat, the tile's pixels met in diagonal order, each lane's sums
                                     kept in registers and added once per (tile, splat).  Same
                                     gradients within float rounding; it evaluates every pixel of a
                                     tile for every splat, and ran 24 times slower than the default
                                     backward on an 800x800 image of 409,660 splats. */
    GSR_OPT_SPLIT = 8,            /* default 1.  The forward records each pixel's transmittance and the
                                     colour behind every 512th position of a tile's list, and the
                                     backward that follows it on the same context (the same bins, the
                                     same final_T and last_contrib buffers) runs each tile whose work
                                     exceeds a CTA slot's share of the frame's work as segments of a
                                     multiple of 512 positions, each its own CTA from those states, so a
                                     crowded tile no longer runs on alone at the end of the launch.
                                     0: one CTA per tile (same results within float rounding). */
    GSR_OPT_SPLIT_FORWARD = 9     /* default 0; takes effect with GSR_OPT_SPLIT.  1: the forward stops
                                     a list longer than a head of max(1024, half the pairs per CTA slot,
                                     rounded up to a multiple of 512) positions there; if a pixel of the
                                     tile still composites, the rest of the list runs as 512-position
                                     chunks, each its own CTA composited from transmittance 1, and each
                                     pixel's stop is found from the chunks' transmittance products and
                                     replayed from the true transmittance in the chunk that holds it.
                                     Transmittance past the head rounds as a product of chunk products,
                                     so final_T and the colour differ from the unsplit forward by float
                                     rounding, and a stop may move where next_T lies within that
                                     rounding of 1e-4.  It pays on frames with a few crowded tiles (an
                                     800x800 close-up whose longest list holds 33,000 pairs: forward
                                     0.25 -> 0.18 ms) and costs on frames without them, where the chunks
                                     past the heads are mostly behind every pixel's stop (800x800,
                                     409,660 splats, 3.7M pairs: 0.118 -> 0.148 ms). */
};

typedef struct gsr_ctx gsr_ctx;

#define GSR_PAIRS_ON_DEVICE 0xffffffffu  /* gsr_bins.num_pairs: the count stayed on the device */

/* Result of gsr_bin_splats.  The device arrays live in the context's arena and
 * stay valid until the next gsr_bin_splats or gsr_destroy on that context. */
typedef struct gsr_bins {
    const uint64_t *keys;        /* device, [num_pairs], ascending (tile << 32 | depth bits);
                                    equal keys are ordered by splat index */
    const uint32_t *sorted_idx;  /* device, [num_pairs], splat index of each key */
    const uint32_t *tile_ranges; /* device, [2 * tiles_x * tiles_y]: {start, end} per tile,
                                    {0, 0} for an empty tile */
    const uint32_t *tile_order;  /* device, [tiles_x * tiles_y]: every tile index once, longest
                                    lists first (by classes of pair count); the forward
                                    launches its CTAs in this order.  NULL: tile order. */
    const uint32_t *num_pairs_dev; /* device, [2]: the pair count (saturated at 0xffffffff) and the
                                    binning's status, GSR_OK or GSR_ERR_TOO_MANY_PAIRS (the count
                                    exceeded the reserved capacity: every tile range is {0, 0});
                                    valid once the binning's work has run */
    uint32_t num_pairs;          /* host copy of the pair count, or GSR_PAIRS_ON_DEVICE when the
                                    binning did not read it back (gsr_reserve_pairs) */
    int32_t n;                   /* splat count the bins were built from */
    int32_t width, height;       /* image size in pixels */
    int32_t tiles_x, tiles_y;    /* ceil(width / 16), ceil(height / 16) */
} gsr_bins;

/* Creates a context on CUDA device `device`.  Allocates nothing on the GPU
 * until the first gsr_bin_splats.  *out receives the context (NULL on error). */
int gsr_create(gsr_ctx **out, int device);

/* Frees the context and its arena.  Safe on NULL.  Waits for nothing: the
 * caller must make sure no enqueued work still uses the arena. */
void gsr_destroy(gsr_ctx *ctx);

/* Text of the last error on this context ("" if none).  Owned by the context. */
const char *gsr_last_error(const gsr_ctx *ctx);

/* Sets a GSR_OPT_* switch (value 0 or 1).  GSR_ERR_INVALID_ARG for an unknown option. */
int gsr_set_option(gsr_ctx *ctx, int option, int value);

/* Number of kernels this context has launched since it was created. */
uint64_t gsr_launch_count(const gsr_ctx *ctx);

/* Bins n splats for a width x height image
 * ("C0 resident arena + C1 pass skip", section 2 table, C0 and C1).
 *
 *   splats  device, [n] gsr_splat2d (4-byte aligned)
 *   depths  device, [n] float; view-space depth, ordered front (small) to back
 *   out     host struct, filled on success
 *
 * A splat emits one pair per tile of its 3-sigma box, rx = 3 sqrt(c / det),
 * ry = 3 sqrt(a / det), det = a c - b^2, tile range floor((mean -+ r) / 16)
 * clamped to the grid; it emits nothing when a field or its depth is not
 * finite, depth <= 0, a <= 0 or det <= 0, or its box misses the image.  The
 * arena grows (never shrinks) to max(65536, 16 n, 1.5 x previous pairs) pairs
 * as needed: the call reads the pair count back (one synchronisation of
 * `stream`) unless the context has a reservation (gsr_reserve_pairs), with
 * which it reads nothing back.  n == 0 is valid and gives empty bins.
 * Errors: GSR_ERR_INVALID_ARG (null ctx/out, n < 0 or > GSR_MAX_SPLATS,
 * width/height outside [1, GSR_MAX_IMAGE_SIDE], null splats/depths with n > 0),
 * GSR_ERR_TOO_MANY_PAIRS, GSR_ERR_OOM, GSR_ERR_CUDA. */
int gsr_bin_splats(gsr_ctx *ctx, const gsr_splat2d *splats, const float *depths, int32_t n,
                   int32_t width, int32_t height, void *stream, gsr_bins *out);

/* Reserves arena capacity for max_pairs tile pairs and switches the context's
 * binning to a mode that reads nothing back to the host
 * ("C0 resident arena + C1 pass skip", section 2 table, C0: the arena grows and
 * is reused; here it is sized ahead so that no call needs the count on the
 * host).  From the next gsr_bin_splats on:
 *   - the call does not synchronise: the arena holds max(max_pairs, 16 n,
 *     65536) pairs (grown at that call if smaller, which does synchronise),
 *     every kernel takes its key counts from the device, and the radix passes
 *     decide on the device which digits to skip;
 *   - bins->num_pairs is GSR_PAIRS_ON_DEVICE and bins->num_pairs_dev holds the
 *     count and the status once the work has run;
 *   - a call whose pairs exceed the capacity emits nothing: its status is
 *     GSR_ERR_TOO_MANY_PAIRS, every tile range is {0, 0} (the forward then
 *     gives final_T = 1 and no colour, the backward zero gradients), and
 *     gsr_num_pairs reports the count that was needed;
 *   - once the arena has its size, a call allocates nothing and can be
 *     captured in a CUDA graph together with the raster calls.
 * max_pairs = 0 returns to the default mode (the count is read back and the
 * arena grown to it).  GSR_ERR_INVALID_ARG for max_pairs > GSR_MAX_PAIRS. */
int gsr_reserve_pairs(gsr_ctx *ctx, uint64_t max_pairs);

/* The pair count of the last gsr_bin_splats on this context: waits for that
 * call's stream, then reads the count from the device.  GSR_ERR_TOO_MANY_PAIRS
 * (with *out the count that was needed) when that binning exceeded its
 * reservation. */
int gsr_num_pairs(gsr_ctx *ctx, uint32_t *out);

/* Forward rasterization over bins made by gsr_bin_splats from the same splats
 * ("forward/adam audit", sections (a), (b), 3; "A.9 f16 forward", snippet;
 * "W1 warp sparse skip + exp-skip", section 1, W1b).
 *
 * For each pixel, front to back over its tile's sorted range: sigma as above
 * with d = pixel - mean; skip sigma < 0 or sigma >= 5.55;
 * alpha = min(0.999, color_a exp(-sigma)); skip alpha < 1/255;
 * next_T = T (1 - alpha); if next_T < 1e-4 the pixel stops without this splat;
 * otherwise C += rgb alpha T, T = next_T.
 *
 *   out_rgbw      device, [height * width] float4 (16-byte aligned): C and 1 - final_T
 *   final_T       device, [height * width] float
 *   last_contrib  device, [height * width] uint32: 1 + position of the last composited
 *                 splat within the tile's range, 0 if none
 * Errors: GSR_ERR_INVALID_ARG (null pointer, misaligned out_rgbw, n differs from
 * bins->n), GSR_ERR_CUDA. */
int gsr_rasterize_forward(gsr_ctx *ctx, const gsr_splat2d *splats, int32_t n,
                          const gsr_bins *bins, float *out_rgbw, float *final_T,
                          uint32_t *last_contrib, void *stream);

/* Backward rasterization: gradient of L = sum_pixels dl_dout.rgb . out.rgb with
 * respect to every Splat2D field ("M3 per-splat backward", section 1;
 * "W1 warp sparse skip + exp-skip", section 1, W1a).  Each pixel replays its
 * composited splats back to front from final_T, recovering the transmittance in
 * front of splat j as T / (1 - alpha_j).  The w channel of dl_dout is ignored.
 *
 *   dl_dout       device, [height * width] float4 (16-byte aligned)
 *   final_T, last_contrib   the forward's outputs for the same bins
 *   grad          device, [n * 9] float, overwritten; row i holds d/d of splat i's
 *                 fields in gsr_splat2d order
 * Each warp's float partial sums are added with double-precision atomics and
 * converted to float at the end; the order of the adds may vary between runs,
 * so the last bits may too (GSR_OPT_DETERMINISTIC makes them fixed).
 * Errors: as gsr_rasterize_forward. */
int gsr_rasterize_backward(gsr_ctx *ctx, const gsr_splat2d *splats, int32_t n,
                           const gsr_bins *bins, const float *dl_dout, const float *final_T,
                           const uint32_t *last_contrib, float *grad, void *stream);

/* Backward rasterization that allocates nothing.  The pages have no counterpart
 * to this entry point; it exists for callers that cannot call cudaMalloc, for
 * example code whose device memory is all reserved up front by another
 * allocator, or loops that must not stall: cudaMalloc may synchronise the
 * device, and it may fail in the middle of a step.
 *
 * Same arguments, result and errors as gsr_rasterize_backward, computed by the
 * same kernels.  Its double-precision accumulator is a fixed device array of
 * GSR_NOALLOC_MAX_SPLATS * 9 doubles (9 MiB), compiled into the library: every
 * GPU that loads libgsr.so holds it until the process exits.  The caller
 * still owns all inputs and outputs, and the bins come from gsr_bin_splats as
 * usual (which does use the context's arena).
 *   - n > GSR_NOALLOC_MAX_SPLATS is rejected with GSR_ERR_INVALID_ARG.
 *   - The first call on a device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.  A
 *     device reset (cudaDeviceReset) invalidates the address it keeps.
 *   - All calls on a device share the one array, and each call clears the part
 *     it uses before accumulating.  Calls whose work overlaps on the GPU (other
 *     streams, other contexts, other threads) race on it: order them. */
#define GSR_NOALLOC_MAX_SPLATS (1 << 17)
int gsr_rasterize_backward_noalloc(gsr_ctx *ctx, const gsr_splat2d *splats, int32_t n,
                                   const gsr_bins *bins, const float *dl_dout, const float *final_T,
                                   const uint32_t *last_contrib, float *grad, void *stream);

/* Statistics of the last gsr_bin_splats (synchronises its stream).
 * The pairs are ordered by two stable LSD radix sorts: the emitting splats by
 * their 32 depth bits in four 8-bit digits, then the pairs by their tile bits
 * split into tile_digits digits of tile_digit_bits bits each.  A digit that
 * every key shares is skipped ("C0 resident arena + C1 pass skip", section 2,
 * C1).  depth_pass_mask / tile_pass_mask: bit f set when digit f was sorted;
 * radix_passes: their total.  capacity: arena capacity in pairs. */
typedef struct gsr_bin_stats {
    uint32_t num_pairs;
    uint32_t emitting;          /* splats with at least one pair */
    int32_t radix_passes;
    uint32_t depth_pass_mask;
    uint32_t tile_pass_mask;
    int32_t tile_digit_bits;
    int32_t tile_digits;
    uint64_t capacity;
} gsr_bin_stats;
int gsr_get_bin_stats(gsr_ctx *ctx, gsr_bin_stats *out);

/* Projection of n 3-D Gaussians to Splat2D records and depths, the step that
 * makes the rasterizer's input in the trainer the pages profile ("M3 per-splat
 * backward", section 3; "W1 warp sparse skip + exp-skip": color_a is the
 * sigmoid of the opacity logit).  The pages give no formula; this is the
 * standard perspective (EWA) projection:
 *
 *   p = W mean + t,  depth = p.z,  mean2 = (fx p.x / p.z + cx, fy p.y / p.z + cy)
 *   J = [[fx / p.z, 0, -fx p.x / p.z^2], [0, fy / p.z, -fy p.y / p.z^2]]
 *   Sigma2 = (J W R S)(J W R S)^T + eps I,  R = rotation of quat / |quat|,
 *            S = diag(exp(log_scale))
 *   conic (a, b, c): [[a, b], [b, c]] = Sigma2^-1,  rgb copied,
 *   color_a = 1 / (1 + exp(-logit_opacity))
 *
 * A Gaussian with a non-finite field, p.z <= z_near, quat = 0 or a singular
 * Sigma2 is not visible: its Splat2D has mean, conic and color_a 0 (rgb is
 * still copied) and its depth is 0, so gsr_bin_splats emits no pair for it.
 *
 *   gauss   device, [n] gsr_gaussian3d (4-byte aligned)
 *   camera  host; read during the call only
 *   splats  device, [n] gsr_splat2d, overwritten
 *   depths  device, [n] float, overwritten
 * Arrays 16-byte aligned take a vectorised path (same results).  Nothing is
 * allocated.  Errors: GSR_ERR_INVALID_ARG (null ctx or camera; n < 0 or
 * > GSR_MAX_SPLATS; null or misaligned arrays with n > 0; a camera field not
 * finite, z_near <= 0 or eps < 0), GSR_ERR_CUDA. */
int gsr_project_forward(gsr_ctx *ctx, const gsr_gaussian3d *gauss, int32_t n, const gsr_camera *camera,
                        gsr_splat2d *splats, float *depths, void *stream);

/* Backward of gsr_project_forward: the gradient of L with respect to every
 * field of every Gaussian, given dl_dsplat = dL/d(each Splat2D field), for
 * example the grad of gsr_rasterize_backward.  Depth carries no gradient (it
 * only orders the splats).  Gaussians that are not visible get 0 in every
 * field, rgb included.
 *
 *   gauss      device, [n] gsr_gaussian3d, as passed to the forward
 *   dl_dsplat  device, [n * 9] float, in gsr_splat2d field order
 *   dl_dgauss  device, [n * 14] float, overwritten, in gsr_gaussian3d field order
 * Errors: as gsr_project_forward. */
int gsr_project_backward(gsr_ctx *ctx, const gsr_gaussian3d *gauss, int32_t n, const gsr_camera *camera,
                         const float *dl_dsplat, float *dl_dgauss, void *stream);

/* Diagnostic: out[i] = exp(-s[i]) computed by the exponential the raster
 * kernels use for alpha = min(0.999, color_a exp(-sigma)) ("A.9 f16 forward",
 * snippet), for 0 <= s[i] <= 5.55 (the only arguments the kernels pass it).
 *   s, out  device, [n] float (4-byte aligned); n >= 0
 * Enqueued on `stream`; nothing is allocated.  GSR_ERR_INVALID_ARG for a NULL
 * or misaligned pointer or n < 0. */
int gsr_exp_neg(gsr_ctx *ctx, const float *s, float *out, int32_t n, void *stream);

/* Diagnostic: one launch of a kernel of known arithmetic, for measuring the
 * device's FP32 and SFU lane-operation rates (the peaks the raster kernels'
 * roofline is taken against; they are ALU-bound).  The grid is 8 CTAs of 256
 * threads per SM.  Each thread runs iters (rounded up to a multiple of 8)
 * rounds of 16 independent operations:
 *   kind GSR_PEAK_FFMA  fused multiply-adds (x = x a + b), 1 lane operation each;
 *   kind GSR_PEAK_EX2   base-2 exponentials on the SFU (ex2.approx, the
 *                       instruction under the kernels' exp(-sigma)).
 *   sink      device, [1] float; written only in a case that never occurs, so
 *             the compiler keeps the work
 *   lane_ops  host; receives the number of lane operations of the launch
 * Time the launch with events on `stream`; rate = lane_ops / time.  Nothing is
 * allocated.  GSR_ERR_INVALID_ARG for an unknown kind, iters outside
 * [1, 2^24], or a NULL pointer. */
enum { GSR_PEAK_FFMA = 0, GSR_PEAK_EX2 = 1 };
int gsr_peak_kernel(gsr_ctx *ctx, int kind, int32_t iters, float *sink, uint64_t *lane_ops, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GSR_H */
