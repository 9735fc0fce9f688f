/*
 * oracle.c -- plain CPU oracle of the tile-binned 2-D splat rasterizer.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Binning lives here; the
 * per-pixel forward and backward live in raster.inc, which this file
 * instantiates once for float (the pages' precision) and once for double
 * (used by the finite-difference pins).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Binning                                                                   */
/* ------------------------------------------------------------------------ */

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* The 3-sigma axis-aligned box of the splat, mapped to 16x16 tiles.
 *
 * The conic (a, b, c) is the inverse covariance, so Sigma = [[c, -b], [-b, a]] / det
 * with det = a c - b^2, and the box half-extents are 3 sqrt(Sigma_xx) and
 * 3 sqrt(Sigma_yy).  The pages name the keys and the tile grid
 * ("p2-c0-resident-binning", section 2, C1: key = (tile_id << 32) | depth_bits,
 * tile_id < num_tiles) but never print the box rule; the 3-sigma box is the
 * plain reading.  Every operation is a single IEEE float operation (this file is
 * built with -ffp-contract=off).
 */
int orc_tile_rect(const float *s, float depth, int32_t tiles_x, int32_t tiles_y, int32_t rect[4])
{
    for (int k = 0; k < 9; ++k)
        if (!isfinite(s[k])) return 0;
    if (!isfinite(depth) || !(depth > 0.0f)) return 0;
    float a = s[2], b = s[3], c = s[4];
    float det = a * c - b * b;
    if (!(a > 0.0f) || !(det > 0.0f)) return 0;
    float sxx = c / det;
    float syy = a / det;
    float rx = 3.0f * sqrtf(sxx);
    float ry = 3.0f * sqrtf(syy);
    float fx0 = (s[0] - rx) * 0.0625f;
    float fx1 = (s[0] + rx) * 0.0625f;
    float fy0 = (s[1] - ry) * 0.0625f;
    float fy1 = (s[1] + ry) * 0.0625f;
    int32_t tx0 = (int32_t)floorf(clampf(fx0, -1.0f, (float)tiles_x));
    int32_t tx1 = (int32_t)floorf(clampf(fx1, -1.0f, (float)tiles_x));
    int32_t ty0 = (int32_t)floorf(clampf(fy0, -1.0f, (float)tiles_y));
    int32_t ty1 = (int32_t)floorf(clampf(fy1, -1.0f, (float)tiles_y));
    if (tx0 < 0) tx0 = 0;
    if (ty0 < 0) ty0 = 0;
    if (tx1 > tiles_x - 1) tx1 = tiles_x - 1;
    if (ty1 > tiles_y - 1) ty1 = tiles_y - 1;
    if (tx0 > tx1 || ty0 > ty1) return 0;
    rect[0] = tx0; rect[1] = ty0; rect[2] = tx1; rect[3] = ty1;
    return 1;
}

static uint32_t float_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

int64_t orc_count_pairs(const float *splats, const float *depths, int32_t n, int32_t width,
                        int32_t height)
{
    int32_t tiles_x = (width + ORC_TILE - 1) / ORC_TILE;
    int32_t tiles_y = (height + ORC_TILE - 1) / ORC_TILE;
    int64_t total = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t r[4];
        if (orc_tile_rect(splats + 9 * (int64_t)i, depths[i], tiles_x, tiles_y, r))
            total += (int64_t)(r[2] - r[0] + 1) * (int64_t)(r[3] - r[1] + 1);
    }
    return total;
}

typedef struct {
    uint64_t key;
    uint32_t idx;
} orc_pair;

static int cmp_pair(const void *pa, const void *pb)
{
    const orc_pair *a = (const orc_pair *)pa, *b = (const orc_pair *)pb;
    if (a->key != b->key) return a->key < b->key ? -1 : 1;
    if (a->idx != b->idx) return a->idx < b->idx ? -1 : 1;
    return 0;
}

/* Pair emission, sort and tile ranges ("p2-c0-resident-binning", section 2:
 * emit -> radix -> extract; the radix sort is stable, so pairs with equal keys
 * keep emission order, which is ascending splat index because a splat emits at
 * most one pair per tile).  Sorting by (key, splat index) with a comparison sort
 * is the plain definition of that result. */
int64_t orc_bin(const float *splats, const float *depths, int32_t n, int32_t width, int32_t height,
                uint64_t *keys, uint32_t *idx, uint32_t *ranges, int64_t cap)
{
    int32_t tiles_x = (width + ORC_TILE - 1) / ORC_TILE;
    int32_t tiles_y = (height + ORC_TILE - 1) / ORC_TILE;
    int64_t num_tiles = (int64_t)tiles_x * tiles_y;
    int64_t total = orc_count_pairs(splats, depths, n, width, height);
    if (total > cap) return -1;
    orc_pair *pairs = (orc_pair *)malloc((size_t)(total > 0 ? total : 1) * sizeof(orc_pair));
    int64_t p = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t r[4];
        if (!orc_tile_rect(splats + 9 * (int64_t)i, depths[i], tiles_x, tiles_y, r)) continue;
        uint32_t dbits = float_bits(depths[i]);
        for (int32_t ty = r[1]; ty <= r[3]; ++ty)
            for (int32_t tx = r[0]; tx <= r[2]; ++tx) {
                uint64_t tile = (uint64_t)ty * (uint64_t)tiles_x + (uint64_t)tx;
                pairs[p].key = (tile << 32) | (uint64_t)dbits;
                pairs[p].idx = (uint32_t)i;
                ++p;
            }
    }
    qsort(pairs, (size_t)p, sizeof(orc_pair), cmp_pair);
    for (int64_t j = 0; j < p; ++j) {
        keys[j] = pairs[j].key;
        idx[j] = pairs[j].idx;
    }
    free(pairs);
    memset(ranges, 0, (size_t)num_tiles * 2 * sizeof(uint32_t));
    for (int64_t j = 0; j < p; ++j) {
        uint64_t tile = keys[j] >> 32;
        if (j == 0 || (keys[j - 1] >> 32) != tile) ranges[2 * tile] = (uint32_t)j;
        if (j == p - 1 || (keys[j + 1] >> 32) != tile) ranges[2 * tile + 1] = (uint32_t)(j + 1);
    }
    return p;
}

/* "p2-c0-resident-binning", section 2, C1: with 4-bit digits a 64-bit key needs
 * 16 passes, and the all-zero digits above the tile field can be skipped:
 * min(16, 8 + ceil(bits(num_tiles - 1) / 4)). */
int32_t orc_radix_passes_4bit(uint64_t num_tiles)
{
    uint64_t v = num_tiles > 0 ? num_tiles - 1 : 0;
    int32_t bits = 0;
    while (v) { ++bits; v >>= 1; }
    int32_t p = 8 + (bits + 3) / 4;
    return p < 16 ? p : 16;
}

/* ------------------------------------------------------------------------ */
/* Forward and backward, once per precision                                  */
/* ------------------------------------------------------------------------ */

/* Decisions within their uncertainty met during a replay (dec nullable, at
 * most max kept), and the flips a replay refused because the decision they
 * name was not within its uncertainty. */
typedef struct {
    orc_decision *dec;
    int32_t max, n;
    int64_t refused;
} orc_trace;

static float orc_exp_f32(float x) { return (float)exp((double)x); }
static double orc_exp_f64(double x) { return exp(x); }

#define REAL float
#define SFX(name) name##_f32
#define REAL_EXP orc_exp_f32
#define REAL_ALPHA_MIN (1.0f / 255.0f)
#define REAL_ALPHA_MAX 0.999f
#define REAL_SIGMA_SKIP 5.55f
#define REAL_T_MIN 1e-4f
#define REAL_ULP 5.9604644775390625e-08 /* 2^-24: half an f32 ulp, relative */
#include "raster.inc"
#undef REAL
#undef SFX
#undef REAL_EXP
#undef REAL_ALPHA_MIN
#undef REAL_ALPHA_MAX
#undef REAL_SIGMA_SKIP
#undef REAL_T_MIN
#undef REAL_ULP

#define REAL double
#define SFX(name) name##_f64
#define REAL_EXP orc_exp_f64
#define REAL_ALPHA_MIN (1.0 / 255.0)
#define REAL_ALPHA_MAX 0.999
#define REAL_SIGMA_SKIP 5.55
#define REAL_T_MIN 1e-4
#define REAL_ULP 1.1102230246251565e-16
#include "raster.inc"
#undef REAL
#undef SFX
#undef REAL_EXP
#undef REAL_ALPHA_MIN
#undef REAL_ALPHA_MAX
#undef REAL_SIGMA_SKIP
#undef REAL_T_MIN
#undef REAL_ULP

/* ------------------------------------------------------------------------ */
/* Brute-force forward (float only)                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    uint32_t dbits;
    uint32_t idx;
} orc_depth_order;

static int cmp_depth(const void *pa, const void *pb)
{
    const orc_depth_order *a = (const orc_depth_order *)pa, *b = (const orc_depth_order *)pb;
    if (a->dbits != b->dbits) return a->dbits < b->dbits ? -1 : 1;
    if (a->idx != b->idx) return a->idx < b->idx ? -1 : 1;
    return 0;
}

/* The culling rule without the box: every field finite, depth > 0, a > 0 and
 * det > 0 (the binning's own tests, before its tile rectangle). */
static int splat_valid(const float *s, float depth)
{
    for (int k = 0; k < 9; ++k)
        if (!isfinite(s[k])) return 0;
    if (!isfinite(depth) || !(depth > 0.0f)) return 0;
    float det = s[2] * s[4] - s[3] * s[3];
    return s[2] > 0.0f && det > 0.0f;
}

static void forward_untiled(const float *splats, const float *depths, int32_t n, int32_t width,
                            int32_t height, float *out_rgbw, float *final_T, uint32_t *last,
                            int skip_sigma, int box)
{
    int32_t tiles_x = (width + ORC_TILE - 1) / ORC_TILE;
    int32_t tiles_y = (height + ORC_TILE - 1) / ORC_TILE;
    orc_depth_order *order = (orc_depth_order *)malloc((size_t)(n > 0 ? n : 1) * sizeof *order);
    int32_t *rects = (int32_t *)malloc((size_t)(n > 0 ? n : 1) * 4 * sizeof(int32_t));
    uint8_t *alive = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    for (int32_t i = 0; i < n; ++i) {
        order[i].dbits = float_bits(depths[i]);
        order[i].idx = (uint32_t)i;
        alive[i] = (uint8_t)orc_tile_rect(splats + 9 * (int64_t)i, depths[i], tiles_x, tiles_y,
                                         rects + 4 * (int64_t)i);
        if (!box) {
            /* every pixel of the image admits every valid splat */
            alive[i] = (uint8_t)splat_valid(splats + 9 * (int64_t)i, depths[i]);
            int32_t *r = rects + 4 * (int64_t)i;
            r[0] = 0; r[1] = 0; r[2] = tiles_x - 1; r[3] = tiles_y - 1;
        }
    }
    qsort(order, (size_t)n, sizeof *order, cmp_depth);
    int64_t cnt[3] = {0, 0, 0};
    for (int32_t py = 0; py < height; ++py)
        for (int32_t px = 0; px < width; ++px) {
            int32_t tx = px / ORC_TILE, ty = py / ORC_TILE;
            pix_f32 st;
            pix_init_f32(&st);
            uint32_t pos = 0; /* position within this pixel's (tile's) list */
            for (int32_t k = 0; k < n && !st.done; ++k) {
                uint32_t i = order[k].idx;
                const int32_t *r = rects + 4 * (int64_t)i;
                if (!alive[i] || tx < r[0] || tx > r[2] || ty < r[1] || ty > r[3]) continue;
                composite_f32(&st, splats + 9 * (int64_t)i, i, (float)px, (float)py, pos, 0.0, 0.0,
                              cnt, skip_sigma, 0u, NULL, NULL);
                ++pos;
            }
            int64_t p = (int64_t)py * width + px;
            out_rgbw[4 * p + 0] = st.C[0];
            out_rgbw[4 * p + 1] = st.C[1];
            out_rgbw[4 * p + 2] = st.C[2];
            out_rgbw[4 * p + 3] = 1.0f - st.T;
            final_T[p] = st.T;
            last[p] = st.last;
        }
    free(order);
    free(rects);
    free(alive);
}

void orc_forward_untiled_f32(const float *splats, const float *depths, int32_t n, int32_t width,
                             int32_t height, float *out_rgbw, float *final_T, uint32_t *last)
{
    forward_untiled(splats, depths, n, width, height, out_rgbw, final_T, last, 1, 1);
}

void orc_forward_untiled_noskip_f32(const float *splats, const float *depths, int32_t n,
                                    int32_t width, int32_t height, float *out_rgbw,
                                    float *final_T, uint32_t *last)
{
    forward_untiled(splats, depths, n, width, height, out_rgbw, final_T, last, 0, 1);
}

void orc_forward_untiled_nobox_f32(const float *splats, const float *depths, int32_t n, int32_t width,
                                   int32_t height, float *out_rgbw, float *final_T, uint32_t *last)
{
    forward_untiled(splats, depths, n, width, height, out_rgbw, final_T, last, 1, 0);
}
