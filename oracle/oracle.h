/*
 * oracle.h -- plain CPU oracle of the tile-binned 2-D splat rasterizer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this code; only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no source with the CUDA path.
 *
 * It is written for a reader checking it against the pages by eye: plain
 * loops, the pages' operation order, no blocking or fusion, one pixel and one
 * splat at a time.  Built with -O2 -ffp-contract=off -fno-fast-math so that
 * every float operation rounds on its own, identically on x86-64 and AArch64.
 *
 * A Splat2D record is 9 floats: mean_x, mean_y, conic_a, conic_b, conic_c,
 * color_r, color_g, color_b, color_a ("p3-forward-adam-audit", staging read:
 * a Splat2D is 9 floats, 36 B).  Tiles are 16x16 pixels.
 *
 * Parity status per function (how each is pinned to something other than
 * itself is listed in tests/test_oracle_pins.py):
 *   orc_tile_rect / orc_count_pairs / orc_bin      pinned
 *   orc_forward_f32 / orc_forward_untiled_f32      pinned
 *   orc_backward_f32 / orc_backward_f64            pinned (finite differences)
 *   orc_project_forward / orc_project_backward     pinned (closed forms, invariances,
 *                                                  finite differences); project.c
 */
#ifndef GSR_ORACLE_H
#define GSR_ORACLE_H
#include <stdint.h>

#define ORC_TILE 16

/* counters[0..2] of a forward: evaluations examined, evaluations with
 * 0 <= sigma < 5.55 (an exponential is needed), splats composited.
 * A backward fills the same three for its replay (positions below
 * last_contributor) in counters[0..2]. */
enum { ORC_N_EVAL = 0, ORC_N_EXP = 1, ORC_N_CONTRIB = 2 };

/* Threshold decisions of one evaluation that another correct float
 * implementation may take the other way when the tested value lies within its
 * rounding uncertainty of the threshold: alpha against 1/255, next_T against
 * 1e-4 (the stop), raw = color_a exp(-sigma) against 0.999 (the clamp, which
 * only the gradient sees). */
enum { ORC_DEC_ALPHA = 1, ORC_DEC_STOP = 2, ORC_DEC_CLAMP = 4 };

/* One entry of a flip table: at pixel (py * width + px), the evaluation at
 * position pos of the tile's list takes the decisions in `type` the other way.
 * Tables are sorted by (pixel, pos). */
typedef struct {
    int64_t pixel;
    uint32_t pos;
    uint32_t type;
} orc_flip;

/* A decision met within its uncertainty: margin = distance to the threshold
 * over the uncertainty of the tested value (below 1). */
typedef struct {
    uint32_t pos;
    uint32_t type;
    uint32_t splat;
    float margin;
} orc_decision;

/* Tile rectangle of one splat's 3-sigma box, inclusive [tx0,tx1]x[ty0,ty1].
 * Returns 0 when the splat is culled (non-finite field, depth <= 0,
 * non-positive-definite conic, box off the image). */
int orc_tile_rect(const float *splat, float depth, int32_t tiles_x, int32_t tiles_y,
                  int32_t rect[4]);

/* Number of (tile, splat) pairs the splats emit. */
int64_t orc_count_pairs(const float *splats, const float *depths, int32_t n,
                        int32_t width, int32_t height);

/* Emits keys (tile_id << 32 | depth_bits) with their splat index, sorts them by
 * (key, splat index) and extracts per-tile ranges {start, end} (2 uint32 per
 * tile, {0,0} when empty).  Returns the pair count, or -1 if it exceeds cap. */
int64_t orc_bin(const float *splats, const float *depths, int32_t n, int32_t width,
                int32_t height, uint64_t *keys, uint32_t *idx, uint32_t *ranges,
                int64_t cap);

/* The pages' 4-bit-digit pass count for a key whose tile field spans
 * num_tiles values: min(16, 8 + ceil(bits(num_tiles - 1) / 4)). */
int32_t orc_radix_passes_4bit(uint64_t num_tiles);

/* Forward over the tile lists (idx, ranges).  out_rgbw: 4 per pixel (rgb and
 * w = 1 - final_T); final_T, last (1 + position of the last composited splat
 * within the tile's range, 0 if none).  margin (nullable): per pixel, the
 * smallest ratio of a threshold decision's distance to its rounding
 * uncertainty, given eps_alpha = the relative uncertainty of one exponential
 * and sigma_ulps = the half-ulps of uncertainty of sigma's terms.
 * counters (nullable): 3 int64. */
void orc_forward_f32(const float *splats, const uint32_t *idx, const uint32_t *ranges,
                     int32_t width, int32_t height, float *out_rgbw, float *final_T,
                     uint32_t *last, float *margin, double eps_alpha, double sigma_ulps,
                     int64_t *counters);
void orc_forward_f64(const double *splats, const uint32_t *idx, const uint32_t *ranges,
                     int32_t width, int32_t height, double *out_rgbw, double *final_T,
                     uint32_t *last, float *margin, double eps_alpha, double sigma_ulps,
                     int64_t *counters);

/* Brute-force forward without tile lists: every pixel walks all splats in
 * (depth_bits, index) order and admits a splat iff its tile rectangle holds the
 * pixel's tile. */
void orc_forward_untiled_f32(const float *splats, const float *depths, int32_t n,
                             int32_t width, int32_t height, float *out_rgbw,
                             float *final_T, uint32_t *last);

/* Same as orc_forward_untiled_f32 without the sigma >= 5.55 skip (used to pin
 * that the skip changes nothing when color_a <= 1). */
void orc_forward_untiled_noskip_f32(const float *splats, const float *depths, int32_t n,
                                    int32_t width, int32_t height, float *out_rgbw,
                                    float *final_T, uint32_t *last);

/* Diagnostic: the brute force without the 3-sigma box predicate (every valid
 * splat may reach every pixel); its difference from orc_forward_untiled_f32 is
 * the colour the box truncates (sigma in [4.5, 5.55) lies outside the box). */
void orc_forward_untiled_nobox_f32(const float *splats, const float *depths, int32_t n,
                                   int32_t width, int32_t height, float *out_rgbw,
                                   float *final_T, uint32_t *last);

/* Backward: gradient of L = sum_p sum_ch dl_dout[p][ch] * out[p][ch] (ch = rgb;
 * w carries no gradient) with respect to the 9 Splat2D fields, accumulated in
 * double into grad[n*9] (overwritten).  gabs (nullable, n*9): the sums of the
 * absolute values of the per-pixel terms of each gradient.  knife (nullable, n bytes): set for each
 * splat examined at a pixel whose margin is below 1, or composited with its
 * unclamped alpha within its uncertainty of the 0.999 cap. */
void orc_backward_f32(const float *splats, int32_t n, const uint32_t *idx,
                      const uint32_t *ranges, int32_t width, int32_t height,
                      const float *dl_dout, double *grad, double *gabs, uint8_t *knife,
                      double eps_alpha, double sigma_ulps, int64_t *counters);
void orc_backward_f64(const double *splats, int32_t n, const uint32_t *idx,
                      const uint32_t *ranges, int32_t width, int32_t height,
                      const double *dl_dout, double *grad, double *gabs, uint8_t *knife,
                      double eps_alpha, double sigma_ulps, int64_t *counters);

/* Forced replays.  The same forward and backward with the decisions a flip
 * table names taken the other way, where each lies within its uncertainty
 * (margin < 1 under eps_alpha and sigma_ulps as above); *refused receives the
 * number of flips that named a decision outside it (those are not taken).
 * They show that a difference between another implementation and the oracle
 * is the other outcome of decisions within rounding, and nothing else. */
void orc_forward_forced_f32(const float *splats, const uint32_t *idx, const uint32_t *ranges,
                            int32_t width, int32_t height, const orc_flip *flips, int64_t nflips,
                            float *out_rgbw, float *final_T, uint32_t *last, double eps_alpha,
                            double sigma_ulps, int64_t *refused);
/* One pixel (px, py): out5 = (r, g, b, 1 - final_T, final_T), *last; the
 * decisions within their uncertainty along its (forced) replay in dec[0, *ndec)
 * (at most max_dec). */
void orc_pixel_forced_f32(const float *splats, const uint32_t *idx, const uint32_t *ranges, int32_t width,
                          int32_t height, int32_t px, int32_t py, const orc_flip *flips, int64_t nflips,
                          double eps_alpha, double sigma_ulps, float *out5, uint32_t *last,
                          orc_decision *dec, int32_t max_dec, int32_t *ndec, int64_t *refused);
void orc_backward_forced_f32(const float *splats, int32_t n, const uint32_t *idx, const uint32_t *ranges,
                             int32_t width, int32_t height, const float *dl_dout, const orc_flip *flips,
                             int64_t nflips, double *grad, double *gabs, double eps_alpha, double sigma_ulps,
                             int64_t *refused);
/* The forced backward's gradients (and sums of |terms|) of the splats
 * targets[0, nt) only, row k for targets[k]; it replays only the tiles whose
 * lists hold a target. */
void orc_backward_targets_f32(const float *splats, int32_t n, const uint32_t *idx, const uint32_t *ranges,
                              int32_t width, int32_t height, const float *dl_dout, const orc_flip *flips,
                              int64_t nflips, const uint32_t *targets, int32_t nt, double *grad_t,
                              double *gabs_t, double eps_alpha, double sigma_ulps, int64_t *refused);
/* Splat `target`'s gradient terms at pixel (px, py) under the flips, out9[9]. */
void orc_pixel_backward_forced_f32(const float *splats, const uint32_t *idx, const uint32_t *ranges,
                                   int32_t width, int32_t height, const float *dl_dout, int32_t px, int32_t py,
                                   const orc_flip *flips, int64_t nflips, uint32_t target, double *out9,
                                   double eps_alpha, double sigma_ulps, int64_t *refused);
/* Splat `target`'s own decisions within their uncertainty at every pixel it is
 * evaluated at (flips applied): out[0, *count) as flip entries, with margins. */
void orc_splat_decisions_f32(const float *splats, int32_t n, const uint32_t *idx, const uint32_t *ranges,
                             int32_t width, int32_t height, const orc_flip *flips, int64_t nflips,
                             uint32_t target, double eps_alpha, double sigma_ulps, orc_flip *out,
                             float *margins, int32_t max, int32_t *count);

/* Projection of 3-D Gaussians to Splat2D records and depths, and its backward
 * (project.c).  Doubles.  g: [n][14] (mean xyz, log_scale xyz, quat wxyz,
 * logit_opacity, rgb); cam: [18] (W row-major, t, fx, fy, cx, cy, z_near,
 * eps); splats: [n][9]; dl_dsplat: [n][9]; dl_dg: [n][14]; gabs: NULL or
 * [n][14], the sum of |terms| of each output's last sum. */
void orc_project_forward(const double *g, int32_t n, const double *cam, double *splats, double *depths,
                         uint8_t *visible);
void orc_project_backward(const double *g, int32_t n, const double *cam, const double *dl_dsplat,
                          double *dl_dg, double *gabs);

#endif
