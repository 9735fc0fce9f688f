// raster.cu -- forward and backward tile rasterization.
//
// One 256-thread CTA per 16x16 tile, one thread per pixel ("forward/adam
// audit" (p3-forward-adam-audit), sections (a), (b), (e): 256-thread group per
// tile staging local_batch[256] Splat2D records).  Each batch of the tile's
// sorted range is staged in shared memory in a compute-ready form.
//
// Warps own 8x4-pixel blocks of the tile.  When a splat is staged, the thread
// that stages it also marks which of the 8 blocks the splat can reach at all:
// the set {sigma < bound} is an ellipse, and its axis-aligned and oriented
// bounding boxes (grown by a margin that covers float rounding) are tested
// against each block.  A warp walks only the splats marked for it, found 32 at
// a time with a ballot.  A skipped evaluation could only have been skipped by
// the per-pixel tests as well, so the results are bit-identical with and
// without this culling.
//
// Both kernels evaluate a splat at a pixel through the same inline functions
// (splat_sigma, splat_alpha), so the backward takes exactly the forward's skip
// and stop decisions.
#include <algorithm>
#include <atomic>
#include <string>

#include "internal.cuh"

// Resident CTAs per SM the raster kernels are compiled for (register budget).
#ifndef GSR_FWD_MIN_BLOCKS
#define GSR_FWD_MIN_BLOCKS 5
#endif
#ifndef GSR_BWD_MIN_BLOCKS
#define GSR_BWD_MIN_BLOCKS 4
#endif
// Splats staged per thread and batch: a batch holds 256 x this many splats.
#ifndef GSR_STAGE_PER_THREAD
#define GSR_STAGE_PER_THREAD 2
#endif
#ifndef GSR_BWD_STAGE_PER_THREAD
#define GSR_BWD_STAGE_PER_THREAD 2
#endif
#ifndef GSR_SPLIT_POSITIONS
#define GSR_SPLIT_POSITIONS 512
#endif

namespace gsr {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = kTilePixels / 32;
constexpr int kBatch = kTilePixels * GSR_STAGE_PER_THREAD;  // splats per staged batch
constexpr int kBwdBatch = kTilePixels * GSR_BWD_STAGE_PER_THREAD;
constexpr float kAlphaMin = 1.0f / 255.0f;  // "W1 warp sparse skip + exp-skip", body
constexpr float kAlphaMax = 0.999f;         // "A.9 f16 forward", snippet
constexpr float kSigmaSkip = 5.55f;         // "W1 warp sparse skip + exp-skip", section 1, W1b
constexpr float kTMin = 1e-4f;              // stop once the transmittance would fall below this
// Granularity of the backward's segments of long lists: the forward records
// each pixel's state at every multiple of this many positions of a list, and
// the backward runs segments of a multiple of it, each from the state
// recorded at its end (a multiple of both batch sizes).
constexpr uint32_t kSplit = GSR_SPLIT_POSITIONS;
static_assert(kSplit % kBatch == 0 && kSplit % kBwdBatch == 0, "segments hold whole batches");
// The backward's segments are sized so that the frame's work (the sum over
// tiles of their largest last_contributor) spreads over this many items per
// CTA slot.
#ifndef GSR_SPLIT_ITEMS_PER_SLOT
#define GSR_SPLIT_ITEMS_PER_SLOT 4
#endif
#ifndef GSR_SPLIT_MIN_SEGMENT
#define GSR_SPLIT_MIN_SEGMENT 512
#endif
constexpr int kSplitItemsPerSlot = GSR_SPLIT_ITEMS_PER_SLOT;
// The segment field of the work item of a tile that is not split.
constexpr uint32_t kWholeList = 0xffffffffu;
// The shortest head after which the forward splits a list.
#ifndef GSR_FWD_HEAD_MIN
#define GSR_FWD_HEAD_MIN 1024
#endif
constexpr uint32_t kFwdHeadMin = GSR_FWD_HEAD_MIN;   // a multiple of kSplit
// (the head's last chunk, which starts inside the list, holds the pixel's stop state)
static_assert(kFwdHeadMin % kSplit == 0 && kFwdHeadMin >= 2 * kSplit, "the head holds two chunks at least");
// CTAs per SM of the chunk and replay grids (each loops over the queued items).
#ifndef GSR_FWD_CHUNK_CTAS_PER_SM
#define GSR_FWD_CHUNK_CTAS_PER_SM GSR_FWD_MIN_BLOCKS
#endif
#ifndef GSR_FWD_REPLAY_CTAS_PER_SM
#define GSR_FWD_REPLAY_CTAS_PER_SM (GSR_FWD_MIN_BLOCKS - 1)
#endif
// The head as a fraction of a CTA slot's fair share of the frame's pairs.
#ifndef GSR_FWD_HEAD_SHARE_NUM
#define GSR_FWD_HEAD_SHARE_NUM 1
#endif
#ifndef GSR_FWD_HEAD_SHARE_DEN
#define GSR_FWD_HEAD_SHARE_DEN 2
#endif
constexpr unsigned long long kFwdHeadShareNum = GSR_FWD_HEAD_SHARE_NUM;
constexpr unsigned long long kFwdHeadShareDen = GSR_FWD_HEAD_SHARE_DEN;
constexpr unsigned long long kSplitMinSegment = GSR_SPLIT_MIN_SEGMENT;   // a multiple of kSplit
// ln(255) plus a margin far above the rounding of the exponent path: a lane whose
// sigma exceeds ln(color_a) + this cannot reach alpha >= 1/255.
constexpr float kLn255Margin = 5.5412636f + 1e-3f;

// Staged splat, three 16-byte vectors per batch slot, plus the warp mask.
//   geo = (mean_x, mean_y, a, b)
//   aux = (c, color_a, sigma bound, splat index as bits)
//   rgb = (r, g, b, 0)
// The sigma bound is min(5.55, ln(color_a) + ln 255 + margin): an evaluation
// with sigma at or above it is skipped without computing an exponential.  At
// 5.55 the bound is the pages' exact skip; below it only lanes whose exact alpha
// test would fail are dropped, so the decisions are those of the exact test.
template <int kSize>
struct StagedBatchT {
    float4 geo[kSize];
    float4 aux[kSize];
    float4 rgb[kSize];
    uint32_t mask[kSize];  // bit w: warp w's 8x4 block may see sigma < bound
};
using StagedBatch = StagedBatchT<kBatch>;

// Warp w covers the 8x4 block (w & 1, w >> 1) of the tile; lane l the pixel
// (l & 7, l >> 3) inside it.
__device__ __forceinline__ int pixel_x(int tid) { return ((tid >> 5) & 1) * 8 + (tid & 7); }
__device__ __forceinline__ int pixel_y(int tid) { return (tid >> 6) * 4 + ((tid >> 3) & 3); }

// Which 8x4 blocks of the tile at (x0, y0) the ellipse {sigma < bound} can reach.
//
// A block is kept when it overlaps the ellipse's slab along each of four
// directions: the x and y axes (the ellipse's bounding box) and its two
// principal axes (its oriented bounding box).  For any direction u, the
// ellipse {1/2 d^T Q d < bound} spans |d . u| <= sqrt(2 bound u^T Q^-1 u), so a
// slab test is valid for whatever direction the rounded eigenvector gives, and
// u need not be normalised (both sides scale with |u|).
//
// The computed sigma may be off by a few roundings of its terms, at most
// 8u (|a| + |c| + 2|b|) / lambda_min relative, and the slab widths carry errors
// of the same order, so every half-width is grown by far more than that
// (plus 1e-3 relative and 1e-3 px); a conic too ill-conditioned for that bound
// to be small is not culled at all.
template <bool kCull>
__device__ __forceinline__ uint32_t block_mask(float mx, float my, float a, float b, float c,
                                               float bound, int x0, int y0)
{
    if (!kCull) return 0xffu;
    if (!(bound > 0.0f)) return 0u;
    const float det = a * c - b * b;
    const float half_tr = 0.5f * (a + c);
    const float rad = sqrtf(0.25f * (a - c) * (a - c) + b * b);
    const float lam_min = half_tr - rad;
    const float rel = 2e-6f * (fabsf(a) + fabsf(c) + 2.0f * fabsf(b)) / lam_min + 1e-3f;
    if (!(det > 0.0f) || !(lam_min > 0.0f) || !(rel < 0.25f)) return 0xffu;
    const float grow = 1.0f + rel;
    const float two_b_det = 2.0f * bound / det;
    const float rx = sqrtf(two_b_det * c) * grow + 1e-3f;
    const float ry = sqrtf(two_b_det * a) * grow + 1e-3f;
    // Principal direction of the largest eigenvalue (a root of the
    // characteristic polynomial), from the better-conditioned of the two
    // forms; v is u rotated by 90 degrees.
    const float lam_max = half_tr + rad;
    const float ux = a >= c ? lam_max - c : b;
    const float uy = a >= c ? b : lam_max - a;
    const float vx = -uy, vy = ux;
    // Half-widths of the ellipse's slabs along u and v, plus the half-extent of
    // an 8x4 block (pixel centres x0..x0+7, y0..y0+3) along each.
    // A quadratic form that rounds below zero, or overflows, gives NaN or
    // infinity here, and the slab tests below then keep the block.
    const float su = sqrtf(two_b_det * (c * ux * ux - 2.0f * b * ux * uy + a * uy * uy));
    const float sv = sqrtf(two_b_det * (c * vx * vx - 2.0f * b * vx * vy + a * vy * vy));
    const float nu = fabsf(ux) + fabsf(uy), nv = fabsf(vx) + fabsf(vy);
    const float lim_u = su * grow + 3.5f * fabsf(ux) + 1.5f * fabsf(uy) + 1e-3f * nu;
    const float lim_v = sv * grow + 3.5f * fabsf(vx) + 1.5f * fabsf(vy) + 1e-3f * nv;
    // Block centre minus mean, projected on u and v, for block 0; the other
    // blocks are offset by (8, 0) and (0, 4) steps.
    const float cx = (float)x0 + 3.5f - mx, cy = (float)y0 + 1.5f - my;
    const float pu0 = cx * ux + cy * uy, pv0 = cx * vx + cy * vy;
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const float bx0 = (float)(x0 + (w & 1) * 8), by0 = (float)(y0 + (w >> 1) * 4);
        const float ox = (float)((w & 1) * 8), oy = (float)((w >> 1) * 4);
        const bool box = (mx - rx <= bx0 + 7.0f) && (mx + rx >= bx0) && (my - ry <= by0 + 3.0f) &&
                         (my + ry >= by0);
        const bool slab_u = !(fabsf(pu0 + ox * ux + oy * uy) > lim_u);  // NaN keeps the block
        const bool slab_v = !(fabsf(pv0 + ox * vx + oy * vy) > lim_v);
        m |= (box && slab_u && slab_v) ? (1u << w) : 0u;
    }
    return m;
}

template <bool kCull, int kSize>
__device__ __forceinline__ void stage_splat(StagedBatchT<kSize> &sb, int slot, const float *__restrict__ splats,
                                            uint32_t idx, int x0, int y0)
{
    const float *s = splats + 9 * (size_t)idx;
    const float mx = __ldg(s + 0), my = __ldg(s + 1);
    const float a = __ldg(s + 2), b = __ldg(s + 3), c = __ldg(s + 4);
    const float r = __ldg(s + 5), g = __ldg(s + 6), bl = __ldg(s + 7);
    const float o = __ldg(s + 8);
    const float bound = fminf(kSigmaSkip, __logf(o) + kLn255Margin);
    sb.geo[slot] = make_float4(mx, my, a, b);
    sb.aux[slot] = make_float4(c, o, bound, __uint_as_float(idx));
    sb.rgb[slot] = make_float4(r, g, bl, 0.0f);
    sb.mask[slot] = block_mask<kCull>(mx, my, a, b, c, bound, x0, y0);
}

// sigma = 1/2 (a dx^2 + c dy^2) + b dx dy, evaluated in exactly that order with
// one rounding per operation (no contraction), so every implementation that
// follows the formula's order gets the same bits.
__device__ __forceinline__ float splat_sigma(const float4 geo, const float c, float px, float py,
                                             float &dx, float &dy)
{
    dx = __fsub_rn(px, geo.x);
    dy = __fsub_rn(py, geo.y);
    const float q = __fadd_rn(__fmul_rn(__fmul_rn(geo.z, dx), dx), __fmul_rn(__fmul_rn(c, dy), dy));
    return __fadd_rn(__fmul_rn(0.5f, q), __fmul_rn(__fmul_rn(geo.w, dx), dy));
}

// exp(-s) for 0 <= s <= 5.55 as 2^(-s log2 e), by Cody and Waite's argument
// splitting: log2 e = L2E + L2E_LO with L2E the float nearest to it, the product
// t = -s L2E rounded, and its rounding error plus -s L2E_LO (an FMA and a
// product) kept as r, so t + r carries -s log2 e to well below an ulp.  2^t is
// the hardware base-2 approximation, and 2^(t + r) = 2^t (1 + r ln 2) to first
// order (|r| < 2^-21).  Over every float s in [0, 5.55] the result is within
// 3 ulp (relative 2e-7) of the correctly rounded exp(-s).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float exp_neg(float s)
{
    constexpr float L2E = 1.44269502f;               // log2(e) rounded to float
    constexpr float L2E_LO = 1.925963033500011e-08f;  // log2(e) - L2E
    constexpr float LN2 = 0.693147182f;
    const float t = __fmul_rn(-s, L2E);
    const float r = __fadd_rn(__fmaf_rn(-s, L2E, -t), __fmul_rn(-s, L2E_LO));
    const float e = ex2_approx(t);
    return __fmaf_rn(e, __fmul_rn(r, LN2), e);
}

// alpha = min(0.999, color_a exp(-sigma)) ("A.9 f16 forward", snippet); also
// returns exp(-sigma) and the unclamped product for the backward.  The
// exponential must be accurate to a few ulp: a deep pixel's colour error grows
// with the sum of its alphas times the per-splat alpha error, and the 1e-5
// forward tolerance leaves no room for a plain hardware approximation, whose
// error grows with the argument.
__device__ __forceinline__ float splat_alpha(float sigma, float o, float &e, float &raw)
{
    e = exp_neg(sigma);
    raw = __fmul_rn(o, e);
    return fminf(kAlphaMax, raw);
}

// --- forward ---------------------------------------------------------------

// Slot of the per-pixel record at position pos of a tile's list, for pos a
// multiple of kSplit with 0 < pos < the list's length: (list start + pos) /
// kSplit.  Two such positions of different lists are more than kSplit apart,
// so their slots differ, and a buffer of pairs / kSplit + 1 slots holds them
// all.  Boundary states live at their boundary's slot; the forward split's
// chunk records at the slot of the chunk's start.
__device__ __forceinline__ size_t bnd_slot(uint32_t list_start, uint32_t pos)
{
    return (size_t)((list_start + pos) / kSplit);
}

// The forward split of crowded tiles.  A list longer than a head of H
// positions stops there in k_forward; if some pixel of the tile is still
// compositing, the rest of the list runs as chunks of kSplit positions, each
// its own CTA, composited from T = 1 (k_forward_chunk), and k_forward_replay
// then finds each pixel's stop from the chunks' transmittance products,
// replays the chunk holding it from the true transmittance, and assembles the
// tile.  H is half a CTA slot's fair share of the frame's pairs, rounded up
// to a multiple of kSplit, and at least kFwdHeadMin.
struct FwdSplit {
    float4 *chunk;             // [slots x 256]: per chunk (colour, transmittance product) from T = 1
    uint32_t *last;            // [slots x 256]: per chunk its last composite (0: none); at the head's
                               // end the pixel's stop: kStopInHead, kNoStop or the chunk that holds it
    uint2 *items;              // (tile, chunk) of every chunk past the head of an unfinished tile
    uint32_t *queue;           // [0] the items' count, [1] replay CTAs finished (both cleared after)
    uint32_t *ticket;          // [tiles] items of the tile finished (cleared after each kernel)
    const uint32_t *pairs_dev; // the frame's pair count on the device, or nullptr
    uint32_t pairs_host;       // the count when pairs_dev is nullptr
    uint32_t bound;            // capacity of items
    int slots;                 // CTA slots of the forward (SMs x resident CTAs)
};

constexpr uint32_t kStopInHead = 0xffffffffu;   // the pixel stopped within the head
constexpr uint32_t kNoStop = 0xfffffffeu;       // the pixel composites to the list's end

// The pixel's stop state lives in the chunk-last record of the head's final
// chunk, which no chunk item uses (chunk items start at the head).
__device__ __forceinline__ size_t head_state_slot(uint32_t list_start, uint32_t head)
{
    return bnd_slot(list_start, head - kSplit);
}

__device__ __forceinline__ uint32_t forward_head(const FwdSplit &fs)
{
    const unsigned long long P = fs.pairs_dev ? (unsigned long long)*fs.pairs_dev : fs.pairs_host;
    const unsigned long long share = (P * kFwdHeadShareNum + (unsigned long long)fs.slots * kFwdHeadShareDen - 1) /
                                     ((unsigned long long)fs.slots * kFwdHeadShareDen);
    const unsigned long long h = max((share + kSplit - 1) / kSplit * kSplit, (unsigned long long)kFwdHeadMin);
    return (uint32_t)min(h, 0x80000000ull);
}

// How composite_batch treats the threshold on the transmittance (the forward's
// own loop, in k_forward, is the rule of kReplay with t_in = 1).
enum CompositeMode {
    kChunkProduct,    // a chunk from T = 1 with no stop of its own: T runs down as the chunk's
                      // transmittance product; a pixel leaves once t_in (a bound on its
                      // transmittance at the chunk's start) times the product falls below the
                      // threshold (the pixel then stops at or before that splat), the product
                      // then including that splat
    kReplay           // the forward's rule, on the transmittance t_in times the running product:
                      // a splat whose next transmittance would fall below the threshold is not
                      // composited and the pixel stops
};

// Composites the staged splats 0..cnt-1 of sb in order into one pixel (T, C,
// last = 1 + the position, offset by pos0, of its last composite).
template <int kMode>
__device__ __forceinline__ void composite_batch(const StagedBatch &sb, int cnt, uint32_t wbit, int lane, float px,
                                                float py, float t_in, float &T, float3 &C, uint32_t &last,
                                                uint32_t pos0, bool &done)
{
    for (int c0 = 0; c0 < cnt; c0 += 32) {
        GSR_CANARY(3);
        uint32_t m = __ballot_sync(kFull, c0 + lane < cnt && (sb.mask[c0 + lane] & wbit));
        while (m) {
            const int j = c0 + __ffs(m) - 1;
            m &= m - 1;
            // Straight-line: every lane evaluates the splat and the predicates
            // take the pixel's skip, stop and composite decisions.
            const float4 geo = sb.geo[j];
            const float4 aux = sb.aux[j];
            const float4 c = sb.rgb[j];
            float dx, dy;
            const float sigma = splat_sigma(geo, aux.x, px, py, dx, dy);
            const bool in_range = !done && sigma >= 0.0f && sigma < aux.z;
            if (!__any_sync(kFull, in_range)) continue;   // no lane can composite: skip the exponential
            float e, raw;
            const float alpha = splat_alpha(in_range ? sigma : 0.0f, aux.y, e, raw);
            const bool ok = in_range && alpha >= kAlphaMin;
            const float next_T = __fmul_rn(T, __fsub_rn(1.0f, alpha));
            const bool stop = ok && __fmul_rn(t_in, next_T) < kTMin;
            const bool comp = ok && !stop;
            const float w = __fmul_rn(alpha, T);
            if (comp) {
                C.x = __fadd_rn(C.x, __fmul_rn(c.x, w));
                C.y = __fadd_rn(C.y, __fmul_rn(c.y, w));
                C.z = __fadd_rn(C.z, __fmul_rn(c.z, w));
                last = pos0 + (uint32_t)j + 1u;
            }
            if (comp || (kMode == kChunkProduct && stop)) T = next_T;
            done = done || stop;
        }
        if (__all_sync(kFull, done)) break;
    }
}

// The colour behind every boundary 1..top of a tile's list (slot(m) = the
// pixel's record at boundary m): each record holds the colour of the segment
// that ends there and the transmittance there; C enters as the colour of the
// part after boundary top.  Turns the colours into suffix sums from the back
// (as the backward accumulates its S) and returns the pixel's colour.  Loads
// go kGroup records at a time ahead of their stores, so a long list does not
// wait for one round trip per boundary.
template <uint32_t kGroup, typename SlotOf>
__device__ __forceinline__ float3 suffix_colours(float4 *bnd, uint32_t top, float3 C, SlotOf slot)
{
    for (uint32_t m = top; m >= 1;) {
        const uint32_t g = min(m, kGroup);
        float4 r[kGroup];
#pragma unroll
        for (uint32_t i = 0; i < kGroup; ++i)
            if (i < g) r[i] = __ldcg(bnd + slot(m - i));
#pragma unroll
        for (uint32_t i = 0; i < kGroup; ++i) {
            if (i < g) {
                bnd[slot(m - i)] = make_float4(C.x, C.y, C.z, r[i].w);
                C = make_float3(__fadd_rn(C.x, r[i].x), __fadd_rn(C.y, r[i].y), __fadd_rn(C.z, r[i].z));
            }
        }
        m -= g;
    }
    return C;
}

// kCut: lists longer than the forward split's head stop there (fs is used);
// otherwise every list runs to its end and fs is ignored.
template <bool kCull, bool kCut>
__global__ void __launch_bounds__(kTilePixels, GSR_FWD_MIN_BLOCKS)
k_forward(const float *__restrict__ splats, const uint32_t *__restrict__ sorted_idx,
          const uint2 *__restrict__ ranges, const uint32_t *__restrict__ order, int width, int height,
          int tiles_x, float4 *__restrict__ out_rgbw, float *__restrict__ final_T, uint32_t *__restrict__ last_out,
          float4 *__restrict__ bnd, FwdSplit fs)
{
    grid_dependency_begin();
    __shared__ StagedBatch sb;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t wbit = 1u << warp;
    const int tile = order ? (int)order[blockIdx.x] : (int)blockIdx.x;
    const int x0 = (tile % tiles_x) * kTile, y0 = (tile / tiles_x) * kTile;
    const int x = x0 + pixel_x(threadIdx.x);
    const int y = y0 + pixel_y(threadIdx.x);
    const bool inside = x < width && y < height;
    const float px = (float)x, py = (float)y;
    const uint2 range = ranges[tile];
    // A list longer than one backward segment records each pixel's state at
    // every segment boundary.  C then holds the colour of the current segment
    // only: it is stored and restarted at each boundary, and the pixel's
    // colour is the sum of its segments' colours, formed at the end.
    const bool record = bnd && range.y - range.x > kSplit;
    // Forward split: a list longer than the head stops after it.
    const uint32_t end = kCut ? range.x + min(range.y - range.x, forward_head(fs)) : range.y;

    float T = 1.0f;
    float3 C = make_float3(0.0f, 0.0f, 0.0f);
    uint32_t last = 0;
    bool done = !inside;
    uint32_t bounds = 0;   // segment boundaries whose state this CTA recorded

    for (uint32_t bstart = range.x; bstart < end; bstart += kBatch) {
        // Every pixel of the tile has stopped: no later splat can change it.
        if (__syncthreads_count(done) == kTilePixels) break;
        // At every multiple of kSplit positions inside the list: the pixel's
        // transmittance and the colour of the segment that ends there.
        if (record && bstart > range.x && (bstart - range.x) % kSplit == 0) {
            bnd[bnd_slot(range.x, bstart - range.x) * kTilePixels + threadIdx.x] = make_float4(C.x, C.y, C.z, T);
            C = make_float3(0.0f, 0.0f, 0.0f);
            ++bounds;
        }
        GSR_CANARY(1);
#pragma unroll
        for (int q = 0; q < GSR_STAGE_PER_THREAD; ++q) {
            const int slot = q * kTilePixels + threadIdx.x;
            const uint32_t pos = bstart + slot;
            if (pos < end) stage_splat<kCull>(sb, slot, splats, __ldg(sorted_idx + pos), x0, y0);
        }
        GSR_CANARY(2);
        __syncthreads();
        const int cnt = (int)min(end - bstart, (uint32_t)kBatch);
        if (__all_sync(kFull, done)) continue;
        for (int c0 = 0; c0 < cnt; c0 += 32) {
            GSR_CANARY(3);
            uint32_t m = __ballot_sync(kFull, c0 + lane < cnt && (sb.mask[c0 + lane] & wbit));
            while (m) {
                const int j = c0 + __ffs(m) - 1;
                m &= m - 1;
                // Straight-line: every lane evaluates the splat and the predicates
                // take the pixel's skip, stop and composite decisions.
                const float4 geo = sb.geo[j];
                const float4 aux = sb.aux[j];
                const float4 c = sb.rgb[j];
                float dx, dy;
                const float sigma = splat_sigma(geo, aux.x, px, py, dx, dy);
                const bool in_range = !done && sigma >= 0.0f && sigma < aux.z;
                if (!__any_sync(kFull, in_range)) continue;   // no lane can composite: skip the exponential
                float e, raw;
                const float alpha = splat_alpha(in_range ? sigma : 0.0f, aux.y, e, raw);
                const bool ok = in_range && alpha >= kAlphaMin;
                const float next_T = __fmul_rn(T, __fsub_rn(1.0f, alpha));
                const bool stop = ok && next_T < kTMin;
                const bool comp = ok && !stop;
                const float w = __fmul_rn(alpha, T);
                if (comp) {
                    C.x = __fadd_rn(C.x, __fmul_rn(c.x, w));
                    C.y = __fadd_rn(C.y, __fmul_rn(c.y, w));
                    C.z = __fadd_rn(C.z, __fmul_rn(c.z, w));
                    T = next_T;
                    last = bstart - range.x + (uint32_t)j + 1u;
                }
                done = done || stop;
            }
            if (__all_sync(kFull, done)) break;
        }
    }
    if constexpr (kCut) {
        // (the tile and its list's end are recomputed rather than kept live
        // through the loop)
        const int tile_id = (y0 / kTile) * tiles_x + x0 / kTile;
        const uint32_t list_end = ranges[tile_id].y;
        if (end != list_end && __syncthreads_count(done) < kTilePixels) {
            // Some pixel still composites at the head's end: record its state
            // there, queue the chunks of the rest of the list, and leave the
            // outputs to the replay.
            const uint32_t len = list_end - range.x, head = end - range.x;
            bnd[bnd_slot(range.x, head) * kTilePixels + threadIdx.x] = make_float4(C.x, C.y, C.z, T);
            fs.last[head_state_slot(range.x, head) * kTilePixels + threadIdx.x] = done ? kStopInHead : 0u;
            if (inside) last_out[(size_t)y * width + x] = last;
            if (threadIdx.x == 0) {
                const uint32_t first = head / kSplit, nch = (len + kSplit - 1) / kSplit - first;
                const uint32_t base = atomicAdd(fs.queue, nch);
                for (uint32_t k = 0; k < nch && base + k < fs.bound; ++k)
                    fs.items[base + k] = make_uint2((uint32_t)tile_id, first + k);
            }
            return;
        }
    }
    // The backward of a segment needs the colour of the splats behind its
    // end: S at a boundary is the sum of the colours of the segments after
    // it, added from the back (as the backward itself accumulates S; a
    // difference of running sums would lose S's digits deep in a long list).
    // The sum over all segments is the pixel's colour.
    for (uint32_t k = bounds; k >= 1; --k) {
        float4 &b = bnd[bnd_slot(range.x, k * kSplit) * kTilePixels + threadIdx.x];
        const float4 c = b;   // the colour of the segment before boundary k
        b = make_float4(C.x, C.y, C.z, c.w);
        C = make_float3(__fadd_rn(C.x, c.x), __fadd_rn(C.y, c.y), __fadd_rn(C.z, c.z));
    }
    if (inside) {
        const size_t p = (size_t)y * width + x;
        out_rgbw[p] = make_float4(C.x, C.y, C.z, __fsub_rn(1.0f, T));
        final_T[p] = T;
        last_out[p] = last;
    }
}

// Once every chunk of a split tile is composited: per pixel, the
// transmittance runs from the head's end through the chunk products; the
// pixel stops inside the first chunk at whose end it falls below the
// threshold.  Each chunk before that gets its colour (its colour from T = 1
// times its start transmittance) and the transmittance at its end in the
// boundary record at its end; the head state records the stop, last_out the
// last composite before it.  A pixel that never stops gets its final colour
// part (the last chunk's) and transmittance in out_rgbw and final_T.  The
// loads do not depend on the stop, so they run ahead of the arithmetic.
__device__ __forceinline__ void prepare_split_pixel(uint2 range, int tile, uint32_t head, size_t p,
                                                    float4 *__restrict__ bnd, const float4 *__restrict__ chunk,
                                                    uint32_t *__restrict__ clast, float4 *__restrict__ out_rgbw,
                                                    float *__restrict__ final_T, uint32_t *__restrict__ last_out)
{
    const uint32_t len = range.y - range.x;
    const uint32_t first = head / kSplit, nchunks = (len + kSplit - 1) / kSplit;
    const size_t hs = head_state_slot(range.x, head) * kTilePixels + threadIdx.x;
    float T = __ldcg(&bnd[bnd_slot(range.x, head) * kTilePixels + threadIdx.x].w);
    if (__ldcg(clast + hs) == kStopInHead) {
        out_rgbw[p] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        final_T[p] = T;
        return;
    }
    uint32_t last = __ldcg(last_out + p);
    uint32_t stop = kNoStop;
    float3 tail = make_float3(0.0f, 0.0f, 0.0f);
#pragma unroll 4
    for (uint32_t k = first; k < nchunks; ++k) {
        const size_t s = bnd_slot(range.x, k * kSplit) * kTilePixels + threadIdx.x;   // the chunk's start
        const float4 r = __ldcg(chunk + s);
        const uint32_t lc = __ldcg(clast + s);
        if (stop == kNoStop) {
            const float Tn = __fmul_rn(T, r.w);
            if (Tn < kTMin) {
                stop = k;
            } else {
                tail = make_float3(__fmul_rn(T, r.x), __fmul_rn(T, r.y), __fmul_rn(T, r.z));
                if (lc) last = k * kSplit + lc;
                T = Tn;
                if (k + 1 < nchunks)   // the boundary at the chunk's end, inside the list
                    bnd[bnd_slot(range.x, (k + 1) * kSplit) * kTilePixels + threadIdx.x] =
                        make_float4(tail.x, tail.y, tail.z, T);
            }
        }
    }
    clast[hs] = stop;
    last_out[p] = last;
    if (stop == kNoStop) {
        out_rgbw[p] = make_float4(tail.x, tail.y, tail.z, 0.0f);
        final_T[p] = T;
    }
}

// The tile's items finished so far, counted after this CTA's writes are
// published; true for the CTA that completes the tile (which clears the count).
__device__ __forceinline__ bool tile_item_done(uint32_t *ticket, int tile, uint32_t items_of_tile, int *s_flag)
{
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t n = atomicAdd(ticket + tile, 1u) + 1u;
        *s_flag = n == items_of_tile;
        if (n == items_of_tile) ticket[tile] = 0;
    }
    __syncthreads();
    const bool last = *s_flag != 0;
    if (last) __threadfence();
    return last;
}

// One chunk past the head of each queued item, composited from T = 1: its
// colour and transmittance product per pixel and its last composite.  The
// last chunk of a tile to finish prepares the tile's replays.
template <bool kCull>
__global__ void __launch_bounds__(kTilePixels, GSR_FWD_MIN_BLOCKS)
k_forward_chunk(const float *__restrict__ splats, const uint32_t *__restrict__ sorted_idx,
                const uint2 *__restrict__ ranges, int width, int height, int tiles_x,
                float4 *__restrict__ out_rgbw, float *__restrict__ final_T, uint32_t *__restrict__ last_out,
                float4 *__restrict__ bnd, FwdSplit fs)
{
    grid_dependency_begin();
    __shared__ StagedBatch sb;
    __shared__ int s_flag;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t wbit = 1u << warp;
    const uint32_t n = min(fs.queue[0], fs.bound);
    const uint32_t head = forward_head(fs), first = head / kSplit;
    for (uint32_t w = blockIdx.x; w < n; w += gridDim.x) {
        if (w > blockIdx.x) __syncthreads();   // the previous item's batch is read
        const uint2 item = fs.items[w];
        const int tile = (int)item.x;
        const int x0 = (tile % tiles_x) * kTile, y0 = (tile / tiles_x) * kTile;
        const int x = x0 + pixel_x(threadIdx.x);
        const int y = y0 + pixel_y(threadIdx.x);
        const bool inside = x < width && y < height;
        const uint2 range = ranges[tile];
        const uint32_t s0 = range.x + item.y * kSplit;
        const int cnt = (int)min(range.y - s0, kSplit);
#pragma unroll
        for (int q = 0; q < GSR_STAGE_PER_THREAD; ++q) {
            const int slot = q * kTilePixels + threadIdx.x;
            if (slot < cnt) stage_splat<kCull>(sb, slot, splats, __ldg(sorted_idx + s0 + slot), x0, y0);
        }
        __syncthreads();
        // The pixel's transmittance at the head's end bounds it at the chunk's
        // start (every later factor is at most 1, and rounding is monotonic);
        // a pixel that stopped within the head has nothing to composite.
        const float t_head = bnd[bnd_slot(range.x, head) * kTilePixels + threadIdx.x].w;
        float T = 1.0f;
        float3 C = make_float3(0.0f, 0.0f, 0.0f);
        uint32_t last = 0;
        bool done = !inside || fs.last[head_state_slot(range.x, head) * kTilePixels + threadIdx.x] == kStopInHead;
        if (!__all_sync(kFull, done))
            composite_batch<kChunkProduct>(sb, cnt, wbit, lane, (float)x, (float)y, t_head, T, C, last, 0u, done);
        const size_t s = bnd_slot(range.x, item.y * kSplit) * kTilePixels + threadIdx.x;   // the chunk's start
        fs.chunk[s] = make_float4(C.x, C.y, C.z, T);
        fs.last[s] = last;
        const uint32_t nch = (range.y - range.x + kSplit - 1) / kSplit - first;
        if (tile_item_done(fs.ticket, tile, nch, &s_flag) && inside)
            prepare_split_pixel(range, tile, head, (size_t)y * width + x, bnd, fs.chunk, fs.last, out_rgbw,
                                final_T, last_out);
    }
}

// Per queued chunk: the pixels that stop inside it replay it from their
// transmittance at its start with the forward's rule, on that start times the
// running product.  The running product repeats the chunk kernel's
// arithmetic splat for splat and rounding is monotonic, so the tested
// transmittance never exceeds the start times the chunk's stored product,
// which fell below the threshold: the replay stops inside the chunk.  The
// last item of a tile to finish assembles the tile's pixels (the suffix pass
// of the forward over all the list's boundaries), and the last CTA of the
// launch clears the queue for the next forward.  No CTA waits on another.
template <bool kCull>
__global__ void __launch_bounds__(kTilePixels, GSR_FWD_MIN_BLOCKS - 1)
k_forward_replay(const float *__restrict__ splats, const uint32_t *__restrict__ sorted_idx,
                 const uint2 *__restrict__ ranges, int width, int height, int tiles_x,
                 float4 *__restrict__ out_rgbw, float *__restrict__ final_T, uint32_t *__restrict__ last_out,
                 float4 *__restrict__ bnd, FwdSplit fs)
{
    grid_dependency_begin();
    __shared__ StagedBatch sb;
    __shared__ int s_flag;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t wbit = 1u << warp;
    const uint32_t n = min(fs.queue[0], fs.bound);
    const uint32_t head = forward_head(fs), first = head / kSplit;
    for (uint32_t w = blockIdx.x; w < n; w += gridDim.x) {
        if (w > blockIdx.x) __syncthreads();   // the previous item's batch is read
        const uint2 item = fs.items[w];
        const int tile = (int)item.x;
        const uint32_t chunk = item.y;
        const int x0 = (tile % tiles_x) * kTile, y0 = (tile / tiles_x) * kTile;
        const int x = x0 + pixel_x(threadIdx.x);
        const int y = y0 + pixel_y(threadIdx.x);
        const bool inside = x < width && y < height;
        const size_t p = (size_t)y * width + x;
        const uint2 range = ranges[tile];
        const size_t hs = head_state_slot(range.x, head) * kTilePixels + threadIdx.x;
        const bool mine = inside && fs.last[hs] == chunk;
        if (__syncthreads_count(mine) > 0) {
            // the transmittance at the chunk's start: the record at its start
            // boundary (the head's own for the first chunk)
            const float t_in = bnd[bnd_slot(range.x, chunk * kSplit) * kTilePixels + threadIdx.x].w;
            const uint32_t s0 = range.x + chunk * kSplit;
            const int cnt = (int)min(range.y - s0, kSplit);
#pragma unroll
            for (int q = 0; q < GSR_STAGE_PER_THREAD; ++q) {
                const int slot = q * kTilePixels + threadIdx.x;
                if (slot < cnt) stage_splat<kCull>(sb, slot, splats, __ldg(sorted_idx + s0 + slot), x0, y0);
            }
            __syncthreads();
            float P = 1.0f;
            float3 C = make_float3(0.0f, 0.0f, 0.0f);
            uint32_t last = 0;
            bool done = !mine;
            if (!__all_sync(kFull, done))
                composite_batch<kReplay>(sb, cnt, wbit, lane, (float)x, (float)y, t_in, P, C, last, 0u, done);
            if (mine) {
                out_rgbw[p] = make_float4(__fmul_rn(t_in, C.x), __fmul_rn(t_in, C.y), __fmul_rn(t_in, C.z), 0.0f);
                final_T[p] = __fmul_rn(t_in, P);
                if (last) last_out[p] = chunk * kSplit + last;
            }
        }
        const uint32_t nch = (range.y - range.x + kSplit - 1) / kSplit - first;
        if (tile_item_done(fs.ticket, tile, nch, &s_flag) && inside) {
            const uint32_t stop = __ldcg(fs.last + hs);
            const uint32_t nchunks = (range.y - range.x + kSplit - 1) / kSplit;
            const uint32_t top = stop == kStopInHead ? first : stop == kNoStop ? nchunks - 1 : stop;
            const float4 o = __ldcg(out_rgbw + p);
            const float T = __ldcg(final_T + p);
            const float3 C = suffix_colours<4>(bnd, top, make_float3(o.x, o.y, o.z), [&](uint32_t m) {
                return bnd_slot(range.x, m * kSplit) * kTilePixels + threadIdx.x;
            });
            out_rgbw[p] = make_float4(C.x, C.y, C.z, __fsub_rn(1.0f, T));
        }
    }
    // The last CTA of the launch clears the queue for the next forward.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(fs.queue + 1, 1u) + 1u == gridDim.x) {
            fs.queue[0] = 0;
            fs.queue[1] = 0;
        }
    }
}

// --- backward --------------------------------------------------------------

// float -> double with integer operations (the FP64 pipe is narrow): exact for
// normal floats and infinities, subnormals flush to a signed zero.
__device__ __forceinline__ double widen(float f)
{
    const uint32_t u = __float_as_uint(f);
    const uint32_t mag = u & 0x7fffffffu;
    uint32_t hi = (mag >> 3) + (896u << 20);
    uint32_t lo = mag << 29;
    const bool small = mag < 0x00800000u;
    hi = small ? 0u : hi;
    lo = small ? 0u : lo;
    hi = mag >= 0x7f800000u ? (0x7ff00000u | ((mag >> 3) & 0xfffffu)) : hi;
    return __hiloint2double((int)(hi | (u & 0x80000000u)), (int)lo);
}

// Deterministic accumulation (GSR_OPT_DETERMINISTIC).  Each warp's partial sum
// x of a gradient component is added to a 64-bit integer accumulator as
// round(x * 2^-E), with E chosen per splat and component group so that the sum
// of every partial the launch can add stays below 2^62 in magnitude (the bounds
// are in k_det_scales).  Integer addition is associative, so the result does not
// depend on the order in which warps add their partials.
//
// round(|x| 2^-E) from the float's bits (ties away from zero); zero and
// subnormal floats give 0.  |x| 2^-E < 2^62 by the choice of E.
__device__ __forceinline__ long long to_fixed(float x, int E)
{
    const uint32_t u = __float_as_uint(x);
    const int ex = (int)((u >> 23) & 0xffu);
    const unsigned long long m = (unsigned long long)((u & 0x7fffffu) | 0x800000u);
    const int sh = ex - 150 - E;  // |x| 2^-E = m 2^sh
    unsigned long long r;
    if (sh >= 0) r = m << min(sh, 39);
    else if (sh > -63) r = (m + (1ull << (-sh - 1))) >> (-sh);
    else r = 0;
    r = ex == 0 ? 0ull : r;
    return (u >> 31) ? -(long long)r : (long long)r;
}

// Group of each gradient component for its fixed-point exponent: 0 the mean
// (components 0, 1), 1 the conic (2..4), 2 the colour (5..7), 3 color_a (8).
__device__ __forceinline__ int det_group(int k) { return k < 2 ? 0 : (k < 5 ? 1 : (k < 8 ? 2 : 3)); }

// Exponent of group grp from a splat's packed exponents (four int16).
__device__ __forceinline__ int det_exponent(uint2 esc, int grp)
{
    const uint32_t w = grp < 2 ? esc.x : esc.y;
    return (int)(int16_t)((grp & 1) ? (w >> 16) : (w & 0xffffu));
}

// Sums the 9 per-lane values over the warp and adds the totals to acc[0..8] in
// one atomic instruction, with 12 shuffles: a transposed butterfly over the
// 16-, 8- and 4-lane exchanges leaves component k (k < 8) summed over those in
// lane group 4k..4k+3 while component 8 rides along as a plain butterfly; at the
// 2-lane exchange the two pair up (lanes with bit 1 clear keep component k,
// the others component 8), and the 1-lane exchange finishes both.  Lanes 4k
// and lane 2 widen their sums to double (with integer operations, off the
// narrow FP64 pipe) and issue the adds.
template <bool kDet>
__device__ __forceinline__ void warp_reduce_add9(float (&v)[9], double *__restrict__ acc, int lane, uint2 esc)
{
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = h16 ? v[i] : v[i + 4];
        const float keep = h16 ? v[i + 4] : v[i];
        w[i] = keep + __shfl_xor_sync(kFull, send, 16);
    }
    float x2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = h8 ? w[i] : w[i + 2];
        const float keep = h8 ? w[i + 2] : w[i];
        x2[i] = keep + __shfl_xor_sync(kFull, send, 8);
    }
    float y = (h4 ? x2[1] : x2[0]) + __shfl_xor_sync(kFull, h4 ? x2[0] : x2[1], 4);
    // component 8 rides along the first three levels, then pairs with y
    float z = v[8];
    z += __shfl_xor_sync(kFull, z, 16);
    z += __shfl_xor_sync(kFull, z, 8);
    z += __shfl_xor_sync(kFull, z, 4);
    const bool h2 = lane & 2;
    float t = (h2 ? z : y) + __shfl_xor_sync(kFull, h2 ? y : z, 2);
    t += __shfl_xor_sync(kFull, t, 1);
    const float mine = t;
    const int k = h2 ? 8 : (lane >> 2);
    if ((lane & 3) == 0 || lane == 2) {
        if (kDet)
            atomicAdd(reinterpret_cast<unsigned long long *>(acc) + k,
                      (unsigned long long)to_fixed(mine, det_exponent(esc, det_group(k))));
        else
            atomicAdd(acc + k, widen(mine));
    }
}

template <bool kWarpSkip, bool kLastContrib, bool kCull, bool kDet>
__global__ void __launch_bounds__(kTilePixels, GSR_BWD_MIN_BLOCKS)
k_backward(const float *__restrict__ splats, const uint32_t *__restrict__ sorted_idx,
           const uint2 *__restrict__ ranges, const uint32_t *__restrict__ order, int width, int height,
           int tiles_x, const float4 *__restrict__ dl_dout, const float *__restrict__ final_T,
           const uint32_t *__restrict__ last_in, double *__restrict__ grad_acc, const uint2 *__restrict__ escale,
           const uint2 *__restrict__ items, const uint32_t *__restrict__ queue, const float4 *__restrict__ bnd)
{
    grid_dependency_begin();
    __shared__ StagedBatchT<kBwdBatch> sb;
    __shared__ uint2 s_esc[kDet ? kBwdBatch : 1];   // fixed-point exponents (deterministic mode)
    __shared__ uint32_t s_wmax[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t wbit = 1u << warp;
    // CTA b takes work items b, b + gridDim.x, ...  Split mode (items set):
    // item w is items[w] = (tile, segment), the positions
    // [segment G, (segment + 1) G) of the tile's list (or all of it), with
    // queue[0] items and G = queue[1] (a multiple of kSplit); the grid holds
    // one CTA per tile, so a CTA takes a second item only when the split
    // makes more items than tiles.  Otherwise CTA b takes tile order[b] (or
    // b), all of it.
    const uint32_t n = items ? __ldg(queue) : 0u;
    const uint32_t seg_len = items ? __ldg(queue + 1) : 0u;
    for (uint32_t w = blockIdx.x; !items || w < n; w += gridDim.x) {
    if (items && w > blockIdx.x) __syncthreads();   // the previous item's shared state is read
    const uint2 item = items ? items[w] : make_uint2(order ? order[w] : w, 0u);
    const int tile = (int)item.x;
    const int x0 = (tile % tiles_x) * kTile, y0 = (tile / tiles_x) * kTile;
    const int x = x0 + pixel_x(threadIdx.x);
    const int y = y0 + pixel_y(threadIdx.x);
    const bool inside = x < width && y < height;
    const float px = (float)x, py = (float)y;
    const uint2 range = ranges[tile];
    const uint32_t len = range.y - range.x;
    const bool whole = !items || item.y == kWholeList;
    const uint32_t s0 = whole ? 0u : item.y * seg_len;
    const uint32_t s1 = whole ? len : min(len, s0 + seg_len);

    float T = 1.0f;
    uint32_t L = 0;
    float3 g = make_float3(0.0f, 0.0f, 0.0f);
    float3 S = make_float3(0.0f, 0.0f, 0.0f);
    if (inside) {
        const size_t p = (size_t)y * width + x;
        T = final_T[p];
        L = min(last_in[p], len);  // a caller's stale last_contrib cannot reach past the range
        if (L > s1) {
            // The pixel composites splats past this segment: start from the
            // state the forward recorded at the segment's end.
            const float4 b = bnd[bnd_slot(range.x, s1) * kTilePixels + threadIdx.x];
            S = make_float3(b.x, b.y, b.z);
            T = b.w;
            L = s1;
        }
        const float4 d = dl_dout[p];
        g = make_float3(d.x, d.y, d.z);
    }
    // Positions at or beyond a pixel's last_contributor were never composited
    // there; a warp stops at its largest, the CTA at the largest of its warps.
    uint32_t warp_end = s1;
    uint32_t cta_end = s1;
    if (kLastContrib) {
        warp_end = __reduce_max_sync(kFull, L);
        if (lane == 0) s_wmax[warp] = warp_end;
        __syncthreads();
        cta_end = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) cta_end = max(cta_end, s_wmax[w]);
    }
    for (int bend = (int)cta_end; bend > (int)s0; bend -= kBwdBatch) {
        const int bstart = max((int)s0, bend - kBwdBatch);
        const int cnt = bend - bstart;
        GSR_CANARY(4);
        __syncthreads();
#pragma unroll
        for (int q = 0; q < GSR_BWD_STAGE_PER_THREAD; ++q) {
            const int slot = q * kTilePixels + threadIdx.x;
            if (slot < cnt) {
                const uint32_t idx = __ldg(sorted_idx + range.x + bstart + slot);
                stage_splat<kCull>(sb, slot, splats, idx, x0, y0);
                if (kDet) s_esc[slot] = escale[idx];
            }
        }
        GSR_CANARY(5);
        __syncthreads();
        const int jlim = min(cnt, (int)warp_end - bstart);  // this warp's positions: j < jlim
        for (int c0 = ((jlim - 1) >> 5) << 5; c0 >= 0 && jlim > 0; c0 -= 32) {
            GSR_CANARY(6);
            uint32_t m = __ballot_sync(kFull, c0 + lane < jlim && (sb.mask[c0 + lane] & wbit));
            while (m) {
                const int bit = 31 - __clz(m);
                m &= ~(1u << bit);
                const int j = c0 + bit;
                const uint32_t rel = (uint32_t)(bstart + j);
                // Straight-line: every lane evaluates the splat and the predicates
                // select (no divergent branches in the warp's loop body).
                const float4 geo = sb.geo[j];
                const float4 aux = sb.aux[j];
                float dx, dy;
                const float sigma = splat_sigma(geo, aux.x, px, py, dx, dy);
                const bool in_range = rel < L && sigma >= 0.0f && sigma < aux.z;
                float e, raw;
                const float alpha = splat_alpha(in_range ? sigma : 0.0f, aux.y, e, raw);
                const bool contrib = in_range && alpha >= kAlphaMin;
                // "W1 warp sparse skip": with no contributing lane nothing changes.
                if (kWarpSkip && !__any_sync(kFull, contrib)) continue;
                const float4 c = sb.rgb[j];
                const float one_m = __fsub_rn(1.0f, alpha);
                const float inv = __fdividef(1.0f, one_m);
                float Tj = T * inv;
                Tj = __fmaf_rn(inv, __fmaf_rn(-one_m, Tj, T), Tj);
                const float aT = alpha * Tj;
                // A lane that does not composite the splat adds zeros: its aT and
                // dRaw are forced to 0 and every term below is a product with one
                // of them (all factors are finite here).
                const float aT_c = contrib ? aT : 0.0f;
                float v[9];
                v[5] = g.x * aT_c;
                v[6] = g.y * aT_c;
                v[7] = g.z * aT_c;
                float dA = g.x * (c.x * Tj - S.x * inv);
                dA = __fmaf_rn(g.y, c.y * Tj - S.y * inv, dA);
                dA = __fmaf_rn(g.z, c.z * Tj - S.z * inv, dA);
                const float dRaw = contrib && raw < kAlphaMax ? dA : 0.0f;
                v[8] = dRaw * e;
                const float dSig = -dRaw * raw;
                const float a = geo.z, bb = geo.w, cc = aux.x;
                v[0] = -dSig * __fmaf_rn(a, dx, bb * dy);
                v[1] = -dSig * __fmaf_rn(bb, dx, cc * dy);
                v[2] = dSig * (0.5f * dx * dx);
                v[3] = dSig * (dx * dy);
                v[4] = dSig * (0.5f * dy * dy);
                if (contrib) {
                    S.x = __fmaf_rn(c.x, aT, S.x);
                    S.y = __fmaf_rn(c.y, aT, S.y);
                    S.z = __fmaf_rn(c.z, aT, S.z);
                    T = Tj;
                }
                warp_reduce_add9<kDet>(v, grad_acc + 9 * (size_t)__float_as_uint(aux.w), lane,
                                       kDet ? s_esc[j] : make_uint2(0u, 0u));
            }
        }
    }
    if (!items) break;
    }
}

// --- per-splat backward ("M3 per-splat backward", section 1) ---------------
//
// The transposed loop nest: one warp per tile, one lane per splat.  The tile's
// composited range is taken back to front in groups of 32 splats; lane l holds
// the splat at position end - 1 - l of the group and meets pixel p at step
// p + l (diagonal scheduling), right after lane l - 1 (the splat behind it) has
// left that pixel's state (T, S) in shared memory.  A lane sums its splat's 9
// gradient components over the tile's 256 pixels in registers, in a fixed
// order, and adds them once per (tile, splat): no reduction across lanes, and
// no atomics within a tile.  Each (pixel, splat) evaluation is the per-pixel
// kernel's: the same skips, the same un-blend of T, the same formulas.
template <bool kDet>
__global__ void __launch_bounds__(32)
k_backward_per_splat(const float *__restrict__ splats, const uint32_t *__restrict__ sorted_idx,
                     const uint2 *__restrict__ ranges, const uint32_t *__restrict__ order, int width, int height,
                     int tiles_x, const float4 *__restrict__ dl_dout, const float *__restrict__ final_T,
                     const uint32_t *__restrict__ last_in, double *__restrict__ grad_acc,
                     const uint2 *__restrict__ escale)
{
    grid_dependency_begin();
    __shared__ float sT[kTilePixels];       // transmittance in front of the next splat to meet the pixel
    __shared__ float sS[3][kTilePixels];    // colour of the splats behind it
    __shared__ float sG[3][kTilePixels];    // dL/dout rgb
    __shared__ uint32_t sL[kTilePixels];    // last_contributor (0 outside the image)
    const int lane = threadIdx.x;
    const int tile = order ? (int)order[blockIdx.x] : (int)blockIdx.x;
    const int x0 = (tile % tiles_x) * kTile, y0 = (tile / tiles_x) * kTile;
    const uint2 range = ranges[tile];
    const uint32_t len = range.y - range.x;
    uint32_t lmax = 0;
    for (int p = lane; p < kTilePixels; p += 32) {
        const int x = x0 + (p & 15), y = y0 + (p >> 4);
        float T = 1.0f;
        uint32_t L = 0;
        float4 d = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (x < width && y < height) {
            const size_t pix = (size_t)y * width + x;
            T = final_T[pix];
            L = min(last_in[pix], len);
            d = dl_dout[pix];
        }
        sT[p] = T;
        sS[0][p] = sS[1][p] = sS[2][p] = 0.0f;
        sG[0][p] = d.x;
        sG[1][p] = d.y;
        sG[2][p] = d.z;
        sL[p] = L;
        lmax = max(lmax, L);
    }
    lmax = __reduce_max_sync(kFull, lmax);
    __syncwarp();
    for (int gend = (int)lmax; gend > 0; gend -= 32) {
        const int pos = gend - 1 - lane;           // this lane's position in the tile's range
        const bool valid = pos >= 0;
        float4 geo = make_float4(0.0f, 0.0f, 0.0f, 0.0f), aux = geo, col = geo;
        uint32_t idx = 0;
        if (valid) {
            idx = __ldg(sorted_idx + range.x + pos);
            const float *sp = splats + 9 * (size_t)idx;
            geo = make_float4(__ldg(sp + 0), __ldg(sp + 1), __ldg(sp + 2), __ldg(sp + 3));
            const float o = __ldg(sp + 8);
            aux = make_float4(__ldg(sp + 4), o, fminf(kSigmaSkip, __logf(o) + kLn255Margin), 0.0f);
            col = make_float4(__ldg(sp + 5), __ldg(sp + 6), __ldg(sp + 7), 0.0f);
        }
        float v[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) v[k] = 0.0f;
        for (int step = 0; step < kTilePixels + 31; ++step) {
            const int p = step - lane;
            if (valid && p >= 0 && p < kTilePixels && (uint32_t)pos < sL[p]) {
                const float px = (float)(x0 + (p & 15)), py = (float)(y0 + (p >> 4));
                float dx, dy;
                const float sigma = splat_sigma(geo, aux.x, px, py, dx, dy);
                if (sigma >= 0.0f && sigma < aux.z) {
                    float e, raw;
                    const float alpha = splat_alpha(sigma, aux.y, e, raw);
                    if (alpha >= kAlphaMin) {
                        const float T = sT[p];
                        const float one_m = __fsub_rn(1.0f, alpha);
                        const float inv = __fdividef(1.0f, one_m);
                        float Tj = T * inv;
                        Tj = __fmaf_rn(inv, __fmaf_rn(-one_m, Tj, T), Tj);
                        const float aT = alpha * Tj;
                        const float gx = sG[0][p], gy = sG[1][p], gz = sG[2][p];
                        const float Sx = sS[0][p], Sy = sS[1][p], Sz = sS[2][p];
                        v[5] += gx * aT;
                        v[6] += gy * aT;
                        v[7] += gz * aT;
                        float dA = gx * (col.x * Tj - Sx * inv);
                        dA = __fmaf_rn(gy, col.y * Tj - Sy * inv, dA);
                        dA = __fmaf_rn(gz, col.z * Tj - Sz * inv, dA);
                        const float dRaw = raw < kAlphaMax ? dA : 0.0f;
                        v[8] += dRaw * e;
                        const float dSig = -dRaw * raw;
                        v[0] += -dSig * __fmaf_rn(geo.z, dx, geo.w * dy);
                        v[1] += -dSig * __fmaf_rn(geo.w, dx, aux.x * dy);
                        v[2] += dSig * (0.5f * dx * dx);
                        v[3] += dSig * (dx * dy);
                        v[4] += dSig * (0.5f * dy * dy);
                        sS[0][p] = __fmaf_rn(col.x, aT, Sx);
                        sS[1][p] = __fmaf_rn(col.y, aT, Sy);
                        sS[2][p] = __fmaf_rn(col.z, aT, Sz);
                        sT[p] = Tj;
                    }
                }
            }
            __syncwarp();
        }
        if (valid) {
            double *acc = grad_acc + 9 * (size_t)idx;
            const uint2 esc = kDet ? escale[idx] : make_uint2(0u, 0u);
#pragma unroll
            for (int k = 0; k < 9; ++k) {
                if (kDet)
                    atomicAdd(reinterpret_cast<unsigned long long *>(acc) + k,
                              (unsigned long long)to_fixed(v[k], det_exponent(esc, det_group(k))));
                else
                    atomicAdd(acc + k, widen(v[k]));
            }
        }
    }
}

// grad = (float)acc, and acc back to zero for the next backward.
__global__ void k_grad_to_float(double *__restrict__ acc, float *__restrict__ grad, size_t count)
{
    grid_dependency_begin();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count;
         i += (size_t)gridDim.x * blockDim.x) {
        grad[i] = (float)acc[i];
        acc[i] = 0.0;
    }
}

// Deterministic mode: the maxima the fixed-point bounds need, one triple per
// block (no atomics): part[3 b], part[3 b + 1] hold the bits of the block's
// largest |dL/dout rgb| and largest |rgb| of a splat whose fields are all
// finite (non-negative floats order like their bits); part[3 b + 2] is set when
// the block saw a non-finite dL/dout.
constexpr int kDetMaxBlocks = 1024;

__global__ void __launch_bounds__(256) k_det_maxima(const float *__restrict__ splats, int n,
                                                    const float4 *__restrict__ dl_dout, size_t npx,
                                                    uint32_t *__restrict__ part)
{
    grid_dependency_begin();
    __shared__ uint32_t s_m[3][8];
    float gm = 0.0f, cm = 0.0f;
    uint32_t nonfinite = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < npx; i += stride) {
        const float4 d = dl_dout[i];
        nonfinite |= !(isfinite(d.x) && isfinite(d.y) && isfinite(d.z));
        gm = fmaxf(gm, fmaxf(fabsf(d.x), fmaxf(fabsf(d.y), fabsf(d.z))));
    }
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < (size_t)n; i += stride) {
        const float *sp = splats + 9 * i;
        bool finite = true;
#pragma unroll
        for (int k = 0; k < 9; ++k) finite &= isfinite(sp[k]);
        if (finite) cm = fmaxf(cm, fmaxf(fabsf(sp[5]), fmaxf(fabsf(sp[6]), fabsf(sp[7]))));
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t gb = __reduce_max_sync(kFull, __float_as_uint(gm));
    const uint32_t cb = __reduce_max_sync(kFull, __float_as_uint(cm));
    const uint32_t nf = __reduce_or_sync(kFull, nonfinite);
    if (lane == 0) {
        s_m[0][warp] = gb;
        s_m[1][warp] = cb;
        s_m[2][warp] = nf;
    }
    __syncthreads();
    if (threadIdx.x < 3) {
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) m = threadIdx.x == 2 ? (m | s_m[2][w]) : max(m, s_m[threadIdx.x][w]);
        part[3 * blockIdx.x + threadIdx.x] = m;
    }
}

// The global maxima from the per-block triples (every thread gets them).
__device__ __forceinline__ void det_global_maxima(const uint32_t *__restrict__ part, int nparts, float &G, float &C,
                                                  bool &nonfinite)
{
    __shared__ uint32_t s_g[3];
    if (threadIdx.x < 32) {
        uint32_t g = 0, c = 0, f = 0;
        for (int b = threadIdx.x; b < nparts; b += 32) {
            g = max(g, part[3 * b]);
            c = max(c, part[3 * b + 1]);
            f |= part[3 * b + 2];
        }
        g = __reduce_max_sync(kFull, g);
        c = __reduce_max_sync(kFull, c);
        f = __reduce_or_sync(kFull, f);
        if (threadIdx.x == 0) {
            s_g[0] = g;
            s_g[1] = c;
            s_g[2] = f;
        }
    }
    __syncthreads();
    G = __uint_as_float(s_g[0]);
    C = __uint_as_float(s_g[1]);
    nonfinite = s_g[2] != 0;
}

// Deterministic mode: per splat, the exponents E of its four gradient groups
// (mean, conic, colour, color_a), packed as int16.  E makes the total of every
// partial the launch can add for the group below 2^62 in magnitude:
//
// One pixel's terms.  With G = max |dL/dout rgb|, C = max |rgb|, and
// alpha <= o' = min(0.999, color_a), the transmittances at most 1 and the
// colour S of the splats behind at most C, |dL/dalpha| <= 3 G C (1 + 1/(1 - o'))
// = A.  A term reaches the conic and mean through dL/dsigma = -dL/dalpha raw,
// raw = color_a e^-sigma < 0.999, and sigma bounds the offsets: 1/2 dx^2 <=
// sigma c / det, 1/2 dy^2 <= sigma a / det, |a dx + b dy| <= sqrt(2 sigma a),
// |b dx + c dy| <= sqrt(2 sigma c); with sigma e^-sigma <= 1/e and
// sqrt(sigma) e^-sigma <= 1 / sqrt(2e) (or raw < 0.999, sigma < 5.55):
//   colour G o';  color_a A;  mean A color_a sqrt(max(a, c) / e);
//   conic A color_a max(c, 2 sqrt(a c), a) / (e det).
// The float sigma is within about 3u lambda_max / lambda_min of the exact one
// (its terms can cancel), far inside the margin while lambda_max / lambda_min
// <= 1e6; a conic worse conditioned than that uses the box instead:
// |dx|, |dy| <= hx, hy, the 3-sigma box radius plus a tile and a pixel.
//
// Partials.  A warp adds 32 pixels' terms, and each of the 8 warps of a tile
// the splat's box reaches adds at most one partial; the total is below
// 2 (margin) x 32 x 8 x tiles x the bound.
__global__ void __launch_bounds__(256) k_det_scales(const float *__restrict__ splats, int n,
                                                    const uint32_t *__restrict__ part, int nparts, int num_tiles,
                                                    uint2 *__restrict__ escale)
{
    // Float arithmetic in the log2 domain (GB300's FP64 pipe is narrow, and
    // nothing overflows there); every bound carries a factor 2 of margin, far
    // above the rounding of these few operations.
    grid_dependency_begin();
    float G, C;
    bool nonfinite;
    det_global_maxima(part, nparts, G, C, nonfinite);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float *sp = splats + 9 * (size_t)i;
    const float a = sp[2], b = sp[3], c = sp[4];
    const float op = fmaxf(0.0f, sp[8]);    // raw = color_a e^-sigma <= op
    const float o = fminf(0.999f, op);       // alpha <= o
    const float l2A = log2f(3.0f * G) + log2f(C) + log2f(1.0f + 1.0f / (1.0f - o));
    const float detf = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, b));
    const float neg_inf = -INFINITY;
    float l2[4] = {neg_inf, neg_inf, log2f(G) + log2f(o), l2A};
    float l2tiles = 0.0f;
    if (detf > 0.0f && a > 0.0f && isfinite(detf) && isfinite(op)) {
        const float rx = 3.0f * sqrtf(c / detf) * 1.0001f, ry = 3.0f * sqrtf(a / detf) * 1.0001f;
        l2tiles = fminf(log2f((float)num_tiles),
                        log2f(floorf(2.0f * rx / 16.0f) + 2.0f) + log2f(floorf(2.0f * ry / 16.0f) + 2.0f));
        const float half_tr = 0.5f * (a + c), rad = sqrtf(0.25f * (a - c) * (a - c) + b * b);
        const float lmax = half_tr + rad, lmin = detf / lmax;
        const float inv_e = 0.36787944f, amax = fmaxf(a, c);
        if (lmin > 0.0f && lmax <= 1e6f * lmin) {
            // raw < 0.999 and sigma < 5.55 also cap raw sqrt(sigma) and raw sigma
            l2[0] = l2A + log2f(fminf(op * sqrtf(amax * inv_e), 0.999f * sqrtf(2.0f * 5.55f * amax)));
            l2[1] = l2A + log2f(fminf(op * inv_e, 0.999f * 5.55f)) +
                    log2f(fmaxf(fmaxf(c, 2.0f * sqrtf(a) * sqrtf(c)), a)) - log2f(detf);
        } else {
            const float hx = rx + 17.0f, hy = ry + 17.0f;
            l2[0] = l2A + log2f(fmaxf(fabsf(a) * hx + fabsf(b) * hy, fabsf(b) * hx + fabsf(c) * hy));
            l2[1] = l2A + fmaxf(fmaxf(2.0f * log2f(hx) - 1.0f, log2f(hx) + log2f(hy)), 2.0f * log2f(hy) - 1.0f);
        }
    }
    // 2 (margin) x 32 lanes x 8 warps per tile x tiles
    const float l2total = 9.0f + l2tiles;
    int E[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float t = l2[k] + l2total + 0.01f;   // log2 of the bound on the total
        E[k] = isfinite(t) ? max(-1100, min(1100, (int)floorf(t) + 1 - 62)) : (t > 0.0f ? 1100 : -200);
    }
    escale[i] = make_uint2(((uint32_t)E[0] & 0xffffu) | ((uint32_t)E[1] << 16),
                           ((uint32_t)E[2] & 0xffffu) | ((uint32_t)E[3] << 16));
}

// Deterministic mode: grad = acc 2^E, and acc back to zero.  A non-finite
// dL/dout makes every gradient NaN.
__global__ void __launch_bounds__(256) k_grad_to_float_det(long long *__restrict__ acc,
                                                           const uint2 *__restrict__ escale,
                                                           const uint32_t *__restrict__ part, int nparts,
                                                           float *__restrict__ grad, size_t count)
{
    grid_dependency_begin();
    float G, C;
    bool nonfinite;
    det_global_maxima(part, nparts, G, C, nonfinite);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t splat = i / 9;
        const int k = (int)(i - splat * 9);
        const int E = det_exponent(escale[splat], det_group(k));
        const float f = ldexpf(__ll2float_rn(acc[i]), E);
        grad[i] = nonfinite ? __int_as_float(0x7fc00000) : f;
        acc[i] = 0;
    }
}

// Work items of the backward: items null, one CTA per tile; else the split's
// (tile, segment) items, queue holding their number and the segment length,
// and bound the most there can be.
struct WorkItems {
    const uint2 *items;
    const uint32_t *queue;
    const float4 *bnd;
    uint32_t bound;
};

template <bool kSkip, bool kLc>
cudaError_t launch_backward_cull(gsr_ctx *ctx, bool cull, int grid, cudaStream_t stream, const float *splats,
                                 const gsr_bins *bins, const uint32_t *order, const float *dl_dout,
                                 const float *final_T, const uint32_t *last_contrib, double *acc,
                                 const uint2 *escale, WorkItems wi)
{
    auto go = [&](auto kernel) {
        return launch_kernel(ctx, kernel, dim3(grid), dim3(kTilePixels), stream, splats, bins->sorted_idx,
                             reinterpret_cast<const uint2 *>(bins->tile_ranges), order, bins->width,
                             bins->height, bins->tiles_x, reinterpret_cast<const float4 *>(dl_dout), final_T,
                             last_contrib, acc, escale, wi.items, wi.queue, wi.bnd);
    };
    if (escale) return cull ? go(k_backward<kSkip, kLc, true, true>) : go(k_backward<kSkip, kLc, false, true>);
    return cull ? go(k_backward<kSkip, kLc, true, false>) : go(k_backward<kSkip, kLc, false, false>);
}

// The backward kernel variant the context's options select, launching tiles
// in `order` (NULL: tile order) and accumulating into acc.
cudaError_t launch_backward(gsr_ctx *ctx, cudaStream_t stream, const float *splats, const gsr_bins *bins,
                            const uint32_t *order, const float *dl_dout, const float *final_T,
                            const uint32_t *last_contrib, double *acc, const uint2 *escale,
                            WorkItems wi = {nullptr, nullptr, nullptr, 0})
{
    const int num_tiles = bins->tiles_x * bins->tiles_y;
    const int grid = num_tiles;   // one CTA per tile, in both modes
    if (ctx->opt_bwd_per_splat) {
        auto go = [&](auto kernel) {   // one CTA per tile
            return launch_kernel(ctx, kernel, dim3(num_tiles), dim3(32), stream, splats, bins->sorted_idx,
                                 reinterpret_cast<const uint2 *>(bins->tile_ranges), order, bins->width,
                                 bins->height, bins->tiles_x, reinterpret_cast<const float4 *>(dl_dout), final_T,
                                 last_contrib, acc, escale);
        };
        return escale ? go(k_backward_per_splat<true>) : go(k_backward_per_splat<false>);
    }
    const bool cull = ctx->opt_warp_cull != 0;
    if (ctx->opt_warp_skip && ctx->opt_last_contrib)
        return launch_backward_cull<true, true>(ctx, cull, grid, stream, splats, bins, order, dl_dout, final_T,
                                                last_contrib, acc, escale, wi);
    if (ctx->opt_warp_skip)
        return launch_backward_cull<true, false>(ctx, cull, grid, stream, splats, bins, order, dl_dout, final_T,
                                                 last_contrib, acc, escale, wi);
    if (ctx->opt_last_contrib)
        return launch_backward_cull<false, true>(ctx, cull, grid, stream, splats, bins, order, dl_dout, final_T,
                                                 last_contrib, acc, escale, wi);
    return launch_backward_cull<false, false>(ctx, cull, grid, stream, splats, bins, order, dl_dout, final_T,
                                              last_contrib, acc, escale, wi);
}

// Per tile: the largest last_contributor of its pixels (one warp per tile), the
// backward's work bound for the tile and the key of its launch order.
__global__ void __launch_bounds__(256)
k_tile_cost(const uint32_t *__restrict__ last, int width, int height, int tiles_x, int num_tiles,
            uint32_t *__restrict__ cost)
{
    grid_dependency_begin();
    const int tile = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (tile >= num_tiles) return;  // whole warps
    const int x0 = (tile % tiles_x) * kTile, y0 = (tile / tiles_x) * kTile;
    const int y = y0 + (lane >> 1), xs = x0 + (lane & 1) * 8;
    uint32_t m = 0;
    if (y < height) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (xs + k < width) m = max(m, last[(size_t)y * width + xs + k]);
    }
    m = __reduce_max_sync(kFull, m);
    if (lane == 0) cost[tile] = m;
}

// 0 for no work, else 1 + floor(8 log2 c): 256 classes a factor 2^(1/8) apart.
__device__ __forceinline__ int work_class(uint32_t c)
{
    return c == 0 ? 0 : min(255, 1 + (int)(8.0f * __log2f((float)c)));
}

// Split mode: the backward's work items in launch order.  A tile is split
// when its largest last_contributor c exceeds a CTA slot's fair share of the
// frame's work (the sum of the tiles' c over the slots): it then gets
// ceil(c / G) items (tile, 0), (tile, 1), ..., G the multiple of kSplit
// nearest above the frame's work over slots x kSplitItemsPerSlot items; any
// other tile with work gets the one item (tile, kWholeList).  In a frame
// without crowded tiles nothing splits.  The items are written in launch
// order, tile by tile, the tiles of larger c first: a counting sort over
// logarithmic classes of c, each class counting its tiles' items.
// queue[0] receives the items' total and queue[1] = G.  One block of 1024
// threads.
__global__ void __launch_bounds__(1024)
k_bwd_plan(const uint32_t *__restrict__ cost, int num_tiles, int slots, uint32_t bound, uint2 *__restrict__ items,
           uint32_t *__restrict__ queue)
{
    grid_dependency_begin();
    __shared__ uint32_t s_hist[256];
    __shared__ unsigned long long s_work;
    __shared__ uint32_t s_items;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        s_work = 0;
        s_items = 0;
    }
    if (threadIdx.x < 256) s_hist[threadIdx.x] = 0;
    __syncthreads();
    unsigned long long work = 0;
    for (int t = threadIdx.x; t < num_tiles; t += 1024) work += cost[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) work += __shfl_xor_sync(kFull, work, o);
    if (lane == 0) atomicAdd(&s_work, work);   // one shared atomic per warp
    __syncthreads();
    const unsigned long long items_wanted = (unsigned long long)slots * kSplitItemsPerSlot;
    const unsigned long long per = (s_work + items_wanted - 1) / items_wanted;
    const unsigned long long g = max((per + kSplit - 1) / kSplit * kSplit, kSplitMinSegment);
    const uint32_t G = (uint32_t)min(g, 0x40000000ull);
    const unsigned long long share = (s_work + slots - 1) / slots;   // a slot's fair share
    // segments of a tile: one unless its work exceeds the share
    auto segments = [&](uint32_t c) -> uint32_t { return c > share ? (c + G - 1) / G : (c ? 1u : 0u); };
    // Each class's item count, and the total.
    uint32_t mine = 0;
    for (int t = threadIdx.x; t < num_tiles; t += 1024) {
        const uint32_t c = cost[t];
        const uint32_t nseg = segments(c);
        if (nseg) atomicAdd(&s_hist[work_class(c)], nseg);
        mine += nseg;
    }
    mine = __reduce_add_sync(kFull, mine);
    if (lane == 0 && mine) atomicAdd(&s_items, mine);
    __syncthreads();
    if (threadIdx.x == 0) {
        queue[0] = min(s_items, bound);
        queue[1] = G;
    }
    // Each class's first place, counted from the largest class down.
    if (threadIdx.x < 32) {
        uint32_t local[8], sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            local[k] = s_hist[255 - (8 * lane + k)];
            sum += local[k];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        uint32_t run = incl - sum;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            s_hist[255 - (8 * lane + k)] = run;
            run += local[k];
        }
    }
    __syncthreads();
    // A tile's items go together to its class's next places (the bound holds
    // by construction; the test keeps the writes inside the buffer regardless).
    for (int t = threadIdx.x; t < num_tiles; t += 1024) {
        const uint32_t c = cost[t];
        const uint32_t nseg = segments(c);
        if (!nseg) continue;
        const uint32_t place = atomicAdd(&s_hist[work_class(c)], nseg);
        for (uint32_t k = 0; k < nseg && place + k < bound; ++k)
            items[place + k] = make_uint2((uint32_t)t, nseg == 1 ? kWholeList : k);
    }
}

}  // namespace

// The pair count of bins, or its bound (the arena's capacity) when it stayed
// on the device.
static uint64_t pairs_bound(const gsr_ctx *ctx, const gsr_bins *bins)
{
    return bins->num_pairs == GSR_PAIRS_ON_DEVICE ? (uint64_t)ctx->cap_pairs : (uint64_t)bins->num_pairs;
}

int rasterize_forward(gsr_ctx *ctx, const float *splats, const gsr_bins *bins, float *out_rgbw,
                      float *final_T, uint32_t *last_contrib, cudaStream_t stream)
{
    const int num_tiles = bins->tiles_x * bins->tiles_y;
    // The boundary states the split backward starts its segments from, and
    // the forward split's chunk states: a slot of 256 pixels per kSplit pairs
    // and one per tile, grown with the pairs.
    float4 *bnd = nullptr;
    FwdSplit fs = {};
    ctx->fwd_bnd_valid = false;
    int rc;
    if (ctx->opt_split) {
        const uint64_t bound = pairs_bound(ctx, bins);
        const size_t slots = (size_t)(bound / kSplit) + 1;
        if (slots > ctx->cap_bnd || !ctx->bnd) {
            if (ctx->bnd) {
                // queued work of an earlier call may still use the old buffer
                if ((rc = cuda_check(ctx, cudaDeviceSynchronize(), "cudaDeviceSynchronize"))) return rc;
                cudaFree(ctx->bnd);
            }
            ctx->bnd = ctx->bnd_chunk = nullptr;
            ctx->bnd_last = nullptr;
            ctx->cap_bnd = 0;
            // boundary states, the forward split's chunk states, their last composites
            if (device_alloc(ctx, (void **)&ctx->bnd, slots * kTilePixels * (2 * sizeof(float4) + sizeof(uint32_t))) !=
                cudaSuccess) {
                cudaGetLastError();
                ctx->bnd = nullptr;
                return fail(ctx, GSR_ERR_OOM, "cudaMalloc failed for the segment boundary states");
            }
            ctx->bnd_chunk = ctx->bnd + slots * kTilePixels;
            ctx->bnd_last = reinterpret_cast<uint32_t *>(ctx->bnd_chunk + slots * kTilePixels);
            ctx->cap_bnd = slots;
        }
        bnd = ctx->bnd;
        if (ctx->opt_split_forward) {
            // At most one item per chunk past a head: fewer than slots.
            if (slots > ctx->cap_fwd_items || (size_t)num_tiles > ctx->cap_fwd_tickets || !ctx->fwd_items) {
                if (ctx->fwd_items) {
                    if ((rc = cuda_check(ctx, cudaDeviceSynchronize(), "cudaDeviceSynchronize"))) return rc;
                    cudaFree(ctx->fwd_items);
                }
                ctx->fwd_items = nullptr;
                ctx->fwd_queue = nullptr;
                ctx->cap_fwd_items = ctx->cap_fwd_tickets = 0;
                const size_t tickets = std::max<size_t>((size_t)num_tiles, 1);
                if (device_alloc(ctx, (void **)&ctx->fwd_items, slots * sizeof(uint2) + (2 + tickets) * sizeof(uint32_t)) !=
                    cudaSuccess) {
                    cudaGetLastError();
                    ctx->fwd_items = nullptr;
                    return fail(ctx, GSR_ERR_OOM, "cudaMalloc failed for the forward split queue");
                }
                ctx->fwd_queue = reinterpret_cast<uint32_t *>(ctx->fwd_items + slots);
                ctx->cap_fwd_items = slots;
                ctx->cap_fwd_tickets = tickets;
                ctx->fwd_queue_dirty = true;
            }
            if (ctx->fwd_queue_dirty) {
                if ((rc = cuda_check(ctx, cudaMemsetAsync(ctx->fwd_queue, 0, (2 + ctx->cap_fwd_tickets) * sizeof(uint32_t),
                                                          stream),
                                     "forward split queue clear")))
                    return rc;
                ctx->fwd_queue_dirty = false;
            }
            const bool on_device = bins->num_pairs == GSR_PAIRS_ON_DEVICE;
            fs.chunk = ctx->bnd_chunk;
            fs.last = ctx->bnd_last;
            fs.items = ctx->fwd_items;
            fs.queue = ctx->fwd_queue;
            fs.ticket = ctx->fwd_queue + 2;
            fs.pairs_dev = on_device ? bins->num_pairs_dev : nullptr;
            fs.pairs_host = on_device ? 0u : bins->num_pairs;
            fs.bound = (uint32_t)std::min<size_t>(ctx->cap_fwd_items, 0xffffffffu);
            fs.slots = ctx->num_sms * GSR_FWD_MIN_BLOCKS;
        }
    }
    const uint2 *ranges = reinterpret_cast<const uint2 *>(bins->tile_ranges);
    float4 *out4 = reinterpret_cast<float4 *>(out_rgbw);
    auto go = [&](auto kernel) {
        return launch_kernel(ctx, kernel, dim3(num_tiles), dim3(kTilePixels), stream, splats, bins->sorted_idx, ranges,
                             bins->tile_order, bins->width, bins->height, bins->tiles_x, out4, final_T, last_contrib,
                             bnd, fs);
    };
    const bool cut = fs.items != nullptr;
    rc = cuda_check(ctx,
                    ctx->opt_warp_cull ? (cut ? go(k_forward<true, true>) : go(k_forward<true, false>))
                                       : (cut ? go(k_forward<false, true>) : go(k_forward<false, false>)),
                    "forward launch");
    if (rc == GSR_OK && fs.items) {
        // The chunks past the heads, then their replays: grids of one wave of
        // CTA slots, looping over the queued items.
        auto wave = [&](int per_sm) {
            return (int)std::max<size_t>(std::min<size_t>(ctx->cap_fwd_items, (size_t)ctx->num_sms * per_sm), 1);
        };
        ctx->fwd_queue_dirty = true;
        auto split_kernel = [&](auto kernel, int grid) {
            return launch_kernel(ctx, kernel, dim3(grid), dim3(kTilePixels), stream, splats, bins->sorted_idx, ranges,
                                 bins->width, bins->height, bins->tiles_x, out4, final_T, last_contrib, bnd, fs);
        };
        const int chunk_grid = wave(GSR_FWD_CHUNK_CTAS_PER_SM), replay_grid = wave(GSR_FWD_REPLAY_CTAS_PER_SM);
        rc = cuda_check(ctx,
                        ctx->opt_warp_cull ? split_kernel(k_forward_chunk<true>, chunk_grid)
                                           : split_kernel(k_forward_chunk<false>, chunk_grid),
                        "forward chunk launch");
        if (rc == GSR_OK)
            rc = cuda_check(ctx,
                            ctx->opt_warp_cull ? split_kernel(k_forward_replay<true>, replay_grid)
                                               : split_kernel(k_forward_replay<false>, replay_grid),
                            "forward replay launch");
        if (rc == GSR_OK) ctx->fwd_queue_dirty = false;
    }
    if (rc == GSR_OK && bnd) {
        ctx->fwd_bnd_valid = true;
        ctx->fwd_bin_call = ctx->bin_calls;
        ctx->fwd_final_T = final_T;
        ctx->fwd_last = last_contrib;
        ctx->fwd_pairs_bound = pairs_bound(ctx, bins);
    }
    return rc;
}

int rasterize_backward(gsr_ctx *ctx, const float *splats, int32_t n, const gsr_bins *bins,
                       const float *dl_dout, const float *final_T, const uint32_t *last_contrib,
                       float *grad, cudaStream_t stream)
{
    const size_t count = (size_t)n * 9;
    int rc;
    if (count > ctx->cap_grad_acc || !ctx->grad_acc) {
        if (ctx->grad_acc) {
            // Queued work may still accumulate into the old buffer.
            if ((rc = cuda_check(ctx, cudaDeviceSynchronize(), "cudaDeviceSynchronize"))) return rc;
            cudaFree(ctx->grad_acc);
        }
        ctx->grad_acc = nullptr;
        ctx->cap_grad_acc = 0;
        const size_t cap = std::max<size_t>(count, 1);
        if (device_alloc(ctx, (void **)&ctx->grad_acc, cap * sizeof(double)) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, GSR_ERR_OOM, "cudaMalloc failed for the gradient accumulator");
        }
        ctx->cap_grad_acc = cap;
        ctx->grad_acc_zero = false;
    }
    // The accumulator is zero between calls: the conversion kernel clears every
    // element it reads.  Only a fresh buffer, or one a failed call left behind,
    // is cleared here.
    if (!ctx->grad_acc_zero) {
        if ((rc = cuda_check(ctx, cudaMemsetAsync(ctx->grad_acc, 0, ctx->cap_grad_acc * sizeof(double), stream),
                             "cudaMemsetAsync")))
            return rc;
        ctx->grad_acc_zero = true;
    }
    // Launch order: tiles with the largest last_contributor (the most work)
    // first, so that no long tile starts late and runs on alone.
    const int num_tiles = bins->tiles_x * bins->tiles_y;
    if ((size_t)num_tiles > ctx->cap_bwd_tiles || !ctx->bwd_tile_cost) {
        if (ctx->bwd_tile_cost) {
            if ((rc = cuda_check(ctx, cudaDeviceSynchronize(), "cudaDeviceSynchronize"))) return rc;
            cudaFree(ctx->bwd_tile_cost);
        }
        ctx->bwd_tile_cost = ctx->bwd_tile_order = nullptr;
        ctx->cap_bwd_tiles = 0;
        const size_t cap = std::max<size_t>((size_t)num_tiles, 1);
        // per tile its cost and the launch order, then the split's item count
        // and segment length
        if (device_alloc(ctx, (void **)&ctx->bwd_tile_cost, (2 * cap + 2) * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            ctx->bwd_tile_cost = nullptr;
            return fail(ctx, GSR_ERR_OOM, "cudaMalloc failed for the backward tile order");
        }
        ctx->bwd_tile_order = ctx->bwd_tile_cost + cap;
        ctx->cap_bwd_tiles = cap;
    }
    uint32_t *queue = ctx->bwd_tile_order + ctx->cap_bwd_tiles;
    // Split mode: long lists run as segments of a multiple of kSplit positions,
    // each from the state this context's forward recorded at its end.  Only
    // over the forward that recorded them: the same bins and the same forward
    // outputs.
    const bool split = ctx->opt_split && !ctx->opt_bwd_per_splat && ctx->fwd_bnd_valid && ctx->bnd &&
                       ctx->fwd_bin_call == ctx->bin_calls && ctx->fwd_final_T == final_T &&
                       ctx->fwd_last == last_contrib;
    size_t item_bound = 0;
    if (split) {
        // at most ceil(len / kSplit) items per tile (num_tiles + pairs / kSplit);
        // and with segments of at least the frame's work W over slots x
        // kSplitItemsPerSlot items, split only in tiles whose work exceeds
        // W / slots (at most slots of them), at most num_tiles + slots x
        // (kSplitItemsPerSlot + 1)
        item_bound = (size_t)num_tiles + std::min<size_t>((size_t)(ctx->fwd_pairs_bound / kSplit),
                                                          (size_t)ctx->num_sms * GSR_BWD_MIN_BLOCKS *
                                                              (kSplitItemsPerSlot + 1));
        if (item_bound > ctx->cap_items || !ctx->bwd_items) {
            if (ctx->bwd_items) {
                if ((rc = cuda_check(ctx, cudaDeviceSynchronize(), "cudaDeviceSynchronize"))) return rc;
                cudaFree(ctx->bwd_items);
            }
            ctx->bwd_items = nullptr;
            ctx->cap_items = 0;
            if (device_alloc(ctx, (void **)&ctx->bwd_items, item_bound * sizeof(uint2)) !=
                cudaSuccess) {
                cudaGetLastError();
                ctx->bwd_items = nullptr;
                return fail(ctx, GSR_ERR_OOM, "cudaMalloc failed for the backward work items");
            }
            ctx->cap_items = item_bound;
        }
    }
    if ((rc = cuda_check(ctx, launch_kernel(ctx, k_tile_cost, dim3((num_tiles + 7) / 8), dim3(256), stream,
                                            last_contrib, bins->width, bins->height, bins->tiles_x, num_tiles,
                                            ctx->bwd_tile_cost),
                         "tile cost launch")))
        return rc;
    if (split) {
        if ((rc = cuda_check(ctx, launch_kernel(ctx, k_bwd_plan, dim3(1), dim3(1024), stream,
                                                (const uint32_t *)ctx->bwd_tile_cost, num_tiles,
                                                ctx->num_sms * GSR_BWD_MIN_BLOCKS, (uint32_t)item_bound, ctx->bwd_items,
                                                queue),
                             "backward plan launch")))
            return rc;
    } else if ((rc = launch_tile_order(ctx, nullptr, ctx->bwd_tile_cost, num_tiles, ctx->bwd_tile_order, stream))) {
        return rc;
    }
    // Deterministic mode: the maxima and the per-splat fixed-point exponents.
    const uint2 *escale = nullptr;
    if (ctx->opt_deterministic) {
        if ((size_t)std::max(n, 1) > ctx->cap_det || !ctx->det_escale) {
            if (ctx->det_escale) {
                if ((rc = cuda_check(ctx, cudaDeviceSynchronize(), "cudaDeviceSynchronize"))) return rc;
                cudaFree(ctx->det_escale);
            }
            ctx->det_escale = nullptr;
            ctx->det_maxima = nullptr;
            ctx->cap_det = 0;
            const size_t cap = std::max<size_t>((size_t)n, 1);
            if (device_alloc(ctx, (void **)&ctx->det_escale, cap * sizeof(uint2) + 3 * kDetMaxBlocks * sizeof(uint32_t)) !=
                cudaSuccess) {
                cudaGetLastError();
                ctx->det_escale = nullptr;
                return fail(ctx, GSR_ERR_OOM, "cudaMalloc failed for the deterministic scales");
            }
            ctx->det_maxima = reinterpret_cast<uint32_t *>(ctx->det_escale + cap);
            ctx->cap_det = cap;
        }
        const size_t npx = (size_t)bins->width * bins->height;
        if ((rc = cuda_check(ctx, launch_kernel(ctx, k_det_maxima, dim3(kDetMaxBlocks), dim3(256), stream, splats,
                                                (int)n, reinterpret_cast<const float4 *>(dl_dout), npx,
                                                ctx->det_maxima),
                             "deterministic maxima launch")))
            return rc;
        if (n > 0 && (rc = cuda_check(ctx, launch_kernel(ctx, k_det_scales, dim3((n + 255) / 256), dim3(256), stream,
                                                         splats, (int)n, (const uint32_t *)ctx->det_maxima,
                                                         kDetMaxBlocks, num_tiles, ctx->det_escale),
                                      "deterministic scales launch")))
            return rc;
        escale = ctx->det_escale;
    }
    ctx->grad_acc_zero = false;
    const WorkItems wi = {split ? ctx->bwd_items : nullptr, queue, split ? ctx->bnd : nullptr,
                          (uint32_t)item_bound};
    if ((rc = cuda_check(ctx, launch_backward(ctx, stream, splats, bins,
                                              split ? nullptr : ctx->bwd_tile_order, dl_dout, final_T,
                                              last_contrib, ctx->grad_acc, escale, wi),
                         "backward launch")))
        return rc;
    if (count > 0) {
        const int blocks = (int)std::min<size_t>((count + 255) / 256, (size_t)ctx->num_sms * 16);
        const cudaError_t e =
            escale ? launch_kernel(ctx, k_grad_to_float_det, dim3(blocks), dim3(256), stream,
                                   reinterpret_cast<long long *>(ctx->grad_acc), escale,
                                   (const uint32_t *)ctx->det_maxima, kDetMaxBlocks, grad, count)
                   : launch_kernel(ctx, k_grad_to_float, dim3(blocks), dim3(256), stream, ctx->grad_acc, grad, count);
        if ((rc = cuda_check(ctx, e, "gradient conversion launch"))) return rc;
    }
    ctx->grad_acc_zero = true;
    return GSR_OK;
}

// --- the exponential on its own (diagnostic) --------------------------------------

namespace {

__global__ void k_exp_neg(const float *__restrict__ s, float *__restrict__ out, int n)
{
    grid_dependency_begin();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) out[i] = exp_neg(s[i]);
}

}  // namespace

int exp_neg_eval(gsr_ctx *ctx, const float *s, float *out, int32_t n, cudaStream_t stream)
{
    const int blocks = (int)std::min<size_t>(((size_t)n + 255) / 256, (size_t)ctx->num_sms * 16);
    return cuda_check(ctx, launch_kernel(ctx, k_exp_neg, dim3(blocks), dim3(256), stream, s, out, (int)n),
                      "exp launch");
}

// --- backward without allocation ---------------------------------------------
//
// For callers that cannot call cudaMalloc, rasterize_backward_noalloc runs the
// same backward kernels with the double-precision accumulator in this fixed
// device array instead of the context's arena.  Every GPU that loads the
// library holds the array until the process exits.

namespace {

__device__ __align__(256) double g_noalloc_grad_acc[(size_t)GSR_NOALLOC_MAX_SPLATS * 9];

// Device address of g_noalloc_grad_acc, looked up once per device (the array's
// name in host code is only a stand-in, not a device pointer).  Atomic: two
// host threads may make their first call on a device at the same time (both
// store the same address).  A device reset invalidates the address.
std::atomic<double *> g_noalloc_ptr[64] = {};

}  // namespace

int rasterize_backward_noalloc(gsr_ctx *ctx, const float *splats, int32_t n, const gsr_bins *bins,
                               const float *dl_dout, const float *final_T,
                               const uint32_t *last_contrib, float *grad, cudaStream_t stream)
{
    if (n > GSR_NOALLOC_MAX_SPLATS)
        return fail(ctx, GSR_ERR_INVALID_ARG,
                    "n = " + std::to_string(n) + " exceeds GSR_NOALLOC_MAX_SPLATS (" +
                        std::to_string(GSR_NOALLOC_MAX_SPLATS) + ")");
    if (ctx->device < 0 || ctx->device >= 64)
        return fail(ctx, GSR_ERR_INVALID_ARG, "device ordinal out of range for the fixed scratch table");
    if (ctx->opt_deterministic)
        return fail(ctx, GSR_ERR_INVALID_ARG, "the deterministic backward needs the context's arena");
    double *acc = g_noalloc_ptr[ctx->device].load(std::memory_order_acquire);
    if (!acc) {
        // First call on this device (the device is current here): find the
        // array's device address.
        void *p = nullptr;
        int rc = cuda_check(ctx, cudaGetSymbolAddress(&p, g_noalloc_grad_acc), "cudaGetSymbolAddress");
        if (rc) return rc;
        acc = static_cast<double *>(p);
        g_noalloc_ptr[ctx->device].store(acc, std::memory_order_release);
    }
    const size_t count = (size_t)n * 9;
    // The array keeps the previous call's sums: clear the part this call uses.
    int rc = cuda_check(ctx, cudaMemsetAsync(acc, 0, count * sizeof(double), stream), "cudaMemsetAsync");
    if (rc) return rc;
    // No allocation here: the forward's launch order (pair count) from the bins.
    if ((rc = cuda_check(ctx, launch_backward(ctx, stream, splats, bins, bins->tile_order, dl_dout, final_T,
                                              last_contrib, acc, nullptr),
                         "backward launch")))
        return rc;
    if (count == 0) return GSR_OK;
    const int blocks = (int)std::min<size_t>((count + 255) / 256, (size_t)ctx->num_sms * 16);
    return cuda_check(ctx, launch_kernel(ctx, k_grad_to_float, dim3(blocks), dim3(256), stream, acc, grad, count),
                      "gradient conversion launch");
}

}  // namespace gsr
