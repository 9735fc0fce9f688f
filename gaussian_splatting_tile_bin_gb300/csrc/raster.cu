// raster.cu -- forward and backward tile rasterization.
//
// One 256-thread CTA per 16x16 tile, one thread per pixel ("forward/adam
// audit" (p3-forward-adam-audit), sections (a), (b), (e): 256-thread group per
// tile staging local_batch[256] Splat2D records).  Each batch of the tile's
// sorted range is staged in shared memory in a compute-ready form (mean, half
// conic, colour, and a per-splat sigma bound); every thread then walks the batch.
//
// Both kernels evaluate a splat at a pixel through the same two inline
// functions (splat_sigma, splat_alpha), so the backward takes exactly the
// forward's skip and stop decisions.
#include <algorithm>
#include <string>

#include "internal.cuh"

namespace gsr {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int SM_BLOCKS_CAP = 152 * 16;     // grid-stride cap for elementwise passes
constexpr float kAlphaMin = 1.0f / 255.0f;  // "W1 warp sparse skip + exp-skip", body
constexpr float kAlphaMax = 0.999f;         // "A.9 f16 forward", snippet
constexpr float kSigmaSkip = 5.55f;         // "W1 warp sparse skip + exp-skip", section 1, W1b
constexpr float kTMin = 1e-4f;              // stop once the transmittance would fall below this
// ln(255) plus a margin far above the rounding of the exponent path: a lane whose
// sigma exceeds ln(color_a) + this cannot reach alpha >= 1/255.
constexpr float kLn255Margin = 5.5412636f + 1e-3f;

// Staged splat, three 16-byte vectors per batch slot.
//   geo = (mean_x, mean_y, a, b)
//   aux = (c, color_a, sigma bound, splat index as bits)
//   rgb = (r, g, b, 0)
// The sigma bound is min(5.55, ln(color_a) + ln 255 + margin): an evaluation
// with sigma at or above it is skipped without computing an exponential.  At
// 5.55 the bound is the pages' exact skip; below it only lanes whose exact alpha
// test would fail are dropped, so the decisions are those of the exact test.
struct StagedBatch {
    float4 geo[kTilePixels];
    float4 aux[kTilePixels];
    float4 rgb[kTilePixels];
};

__device__ __forceinline__ void stage_splat(StagedBatch &sb, int slot, const float *__restrict__ splats,
                                            uint32_t idx)
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

// alpha = min(0.999, color_a exp(-sigma)) ("A.9 f16 forward", snippet); also
// returns exp(-sigma) and the unclamped product for the backward.  expf is the
// accurate exponential (within 2 ulp): a deep pixel's colour error grows with the
// sum of its alphas times the per-splat alpha error, and the 1e-5 forward
// tolerance leaves no room for the approximate one.
__device__ __forceinline__ float splat_alpha(float sigma, float o, float &e, float &raw)
{
    e = expf(-sigma);
    raw = __fmul_rn(o, e);
    return fminf(kAlphaMax, raw);
}

__device__ __forceinline__ int pixel_x(int tid) { return tid & (kTile - 1); }
__device__ __forceinline__ int pixel_y(int tid) { return tid >> 4; }

// --- forward ---------------------------------------------------------------

__global__ void __launch_bounds__(kTilePixels)
k_forward(const float *__restrict__ splats, const uint32_t *__restrict__ sorted_idx,
          const uint2 *__restrict__ ranges, int width, int height, int tiles_x,
          float4 *__restrict__ out_rgbw, float *__restrict__ final_T, uint32_t *__restrict__ last_out)
{
    __shared__ StagedBatch sb;
    const int tile = blockIdx.x;
    const int tx = tile % tiles_x, ty = tile / tiles_x;
    const int x = tx * kTile + pixel_x(threadIdx.x);
    const int y = ty * kTile + pixel_y(threadIdx.x);
    const bool inside = x < width && y < height;
    const float px = (float)x, py = (float)y;
    const uint2 range = ranges[tile];

    float T = 1.0f;
    float3 C = make_float3(0.0f, 0.0f, 0.0f);
    uint32_t last = 0;
    bool done = !inside;

    for (uint32_t bstart = range.x; bstart < range.y; bstart += kTilePixels) {
        // Every pixel of the tile has stopped: no later splat can change it.
        if (__syncthreads_count(done) == kTilePixels) break;
        const uint32_t pos = bstart + threadIdx.x;
        if (pos < range.y) stage_splat(sb, threadIdx.x, splats, __ldg(sorted_idx + pos));
        __syncthreads();
        const int cnt = (int)min(range.y - bstart, (uint32_t)kTilePixels);
        if (!done) {
            for (int j = 0; j < cnt; ++j) {
                const float4 geo = sb.geo[j];
                const float4 aux = sb.aux[j];
                float dx, dy;
                const float sigma = splat_sigma(geo, aux.x, px, py, dx, dy);
                if (!(sigma >= 0.0f) || !(sigma < aux.z)) continue;
                float e, raw;
                const float alpha = splat_alpha(sigma, aux.y, e, raw);
                if (alpha < kAlphaMin) continue;
                const float next_T = __fmul_rn(T, __fsub_rn(1.0f, alpha));
                if (next_T < kTMin) {
                    done = true;
                    break;
                }
                const float w = __fmul_rn(alpha, T);
                const float4 c = sb.rgb[j];
                C.x = __fadd_rn(C.x, __fmul_rn(c.x, w));
                C.y = __fadd_rn(C.y, __fmul_rn(c.y, w));
                C.z = __fadd_rn(C.z, __fmul_rn(c.z, w));
                T = next_T;
                last = bstart - range.x + (uint32_t)j + 1u;
            }
        }
    }
    if (inside) {
        const size_t p = (size_t)y * width + x;
        out_rgbw[p] = make_float4(C.x, C.y, C.z, __fsub_rn(1.0f, T));
        final_T[p] = T;
        last_out[p] = last;
    }
}

// --- backward --------------------------------------------------------------

template <bool kWarpSkip, bool kLastContrib>
__global__ void __launch_bounds__(kTilePixels)
k_backward(const float *__restrict__ splats, const uint32_t *__restrict__ sorted_idx,
           const uint2 *__restrict__ ranges, int width, int height, int tiles_x,
           const float4 *__restrict__ dl_dout, const float *__restrict__ final_T,
           const uint32_t *__restrict__ last_in, double *__restrict__ grad_acc)
{
    __shared__ StagedBatch sb;
    __shared__ uint32_t s_wmax[kTilePixels / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile = blockIdx.x;
    const int tx = tile % tiles_x, ty = tile / tiles_x;
    const int x = tx * kTile + pixel_x(threadIdx.x);
    const int y = ty * kTile + pixel_y(threadIdx.x);
    const bool inside = x < width && y < height;
    const float px = (float)x, py = (float)y;
    const uint2 range = ranges[tile];
    const uint32_t len = range.y - range.x;

    float T = 1.0f;
    uint32_t L = 0;
    float3 g = make_float3(0.0f, 0.0f, 0.0f);
    if (inside) {
        const size_t p = (size_t)y * width + x;
        T = final_T[p];
        L = min(last_in[p], len);  // a caller's stale last_contrib cannot reach past the range
        const float4 d = dl_dout[p];
        g = make_float3(d.x, d.y, d.z);
    }
    // Positions at or beyond a pixel's last_contributor were never composited
    // there; a warp stops at its largest, the CTA at the largest of its warps.
    uint32_t warp_end = len;
    uint32_t cta_end = len;
    if (kLastContrib) {
        warp_end = __reduce_max_sync(kFull, L);
        if (lane == 0) s_wmax[warp] = warp_end;
        __syncthreads();
        cta_end = 0;
#pragma unroll
        for (int w = 0; w < kTilePixels / 32; ++w) cta_end = max(cta_end, s_wmax[w]);
    }
    float3 S = make_float3(0.0f, 0.0f, 0.0f);

    for (int bend = (int)cta_end; bend > 0; bend -= kTilePixels) {
        const int bstart = max(0, bend - kTilePixels);
        const int cnt = bend - bstart;
        __syncthreads();
        if (threadIdx.x < cnt)
            stage_splat(sb, threadIdx.x, splats, __ldg(sorted_idx + range.x + bstart + threadIdx.x));
        __syncthreads();
        const int jhi = min(cnt, (int)warp_end - bstart) - 1;
        for (int j = jhi; j >= 0; --j) {
            const uint32_t rel = (uint32_t)(bstart + j);
            bool contrib = false;
            float v[9];
#pragma unroll
            for (int k = 0; k < 9; ++k) v[k] = 0.0f;
            if (rel < L) {
                const float4 geo = sb.geo[j];
                const float4 aux = sb.aux[j];
                float dx, dy;
                const float sigma = splat_sigma(geo, aux.x, px, py, dx, dy);
                if (sigma >= 0.0f && sigma < aux.z) {
                    float e, raw;
                    const float alpha = splat_alpha(sigma, aux.y, e, raw);
                    if (alpha >= kAlphaMin) {
                        contrib = true;
                        const float4 c = sb.rgb[j];
                        const float one_m = __fsub_rn(1.0f, alpha);
                        const float inv = __fdividef(1.0f, one_m);
                        // Transmittance in front of this splat: the forward's
                        // T_j (1 - alpha) undone with one correctly rounded division,
                        // so a pixel replayed through hundreds of splats drifts by at
                        // most a rounding per splat.
                        const float Tj = __fdiv_rn(T, one_m);
                        const float aT = alpha * Tj;
                        v[5] = g.x * aT;
                        v[6] = g.y * aT;
                        v[7] = g.z * aT;
                        float dA = g.x * (c.x * Tj - S.x * inv);
                        dA = __fmaf_rn(g.y, c.y * Tj - S.y * inv, dA);
                        dA = __fmaf_rn(g.z, c.z * Tj - S.z * inv, dA);
                        S.x = __fmaf_rn(c.x, aT, S.x);
                        S.y = __fmaf_rn(c.y, aT, S.y);
                        S.z = __fmaf_rn(c.z, aT, S.z);
                        const float dRaw = raw < kAlphaMax ? dA : 0.0f;
                        v[8] = dRaw * e;
                        const float dSig = -dRaw * raw;
                        const float a = geo.z, b = geo.w, cc = aux.x;
                        v[0] = -dSig * __fmaf_rn(a, dx, b * dy);
                        v[1] = -dSig * __fmaf_rn(b, dx, cc * dy);
                        v[2] = dSig * (0.5f * dx * dx);
                        v[3] = dSig * (dx * dy);
                        v[4] = dSig * (0.5f * dy * dy);
                        T = Tj;
                    }
                }
            }
            // "W1 warp sparse skip": with no contributing lane every sum is +0.
            if (kWarpSkip && !__any_sync(kFull, contrib)) continue;
#pragma unroll
            for (int k = 0; k < 9; ++k) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(kFull, v[k], o);
            }
            // One atomic per warp, splat and field, accumulated in double: a
            // large splat sums thousands of warp partials of both signs, and in
            // float their order alone moves the result by more than 1e-4.
            if (lane == 0) {
                const uint32_t idx = __float_as_uint(sb.aux[j].w);
                double *gr = grad_acc + 9 * (size_t)idx;
#pragma unroll
                for (int k = 0; k < 9; ++k) atomicAdd(gr + k, (double)v[k]);
            }
        }
    }
}

__global__ void k_grad_to_float(const double *__restrict__ acc, float *__restrict__ grad, size_t count)
{
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count;
         i += (size_t)gridDim.x * blockDim.x)
        grad[i] = (float)acc[i];
}

}  // namespace

int rasterize_forward(gsr_ctx *ctx, const float *splats, const gsr_bins *bins, float *out_rgbw,
                      float *final_T, uint32_t *last_contrib, cudaStream_t stream)
{
    const int num_tiles = bins->tiles_x * bins->tiles_y;
    k_forward<<<num_tiles, kTilePixels, 0, stream>>>(
        splats, bins->sorted_idx, reinterpret_cast<const uint2 *>(bins->tile_ranges), bins->width,
        bins->height, bins->tiles_x, reinterpret_cast<float4 *>(out_rgbw), final_T, last_contrib);
    ++ctx->launches;
    return cuda_check(ctx, cudaGetLastError(), "forward launch");
}

int rasterize_backward(gsr_ctx *ctx, const float *splats, int32_t n, const gsr_bins *bins,
                       const float *dl_dout, const float *final_T, const uint32_t *last_contrib,
                       float *grad, cudaStream_t stream)
{
    const size_t count = (size_t)n * 9;
    if (count > ctx->cap_grad_acc || !ctx->grad_acc) {
        if (ctx->grad_acc) cudaFree(ctx->grad_acc);
        ctx->grad_acc = nullptr;
        ctx->cap_grad_acc = 0;
        if (cudaMalloc(&ctx->grad_acc, count * sizeof(double)) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, GSR_ERR_OOM, "cudaMalloc failed for the gradient accumulator");
        }
        ctx->cap_grad_acc = count;
    }
    int rc = cuda_check(ctx, cudaMemsetAsync(ctx->grad_acc, 0, count * sizeof(double), stream),
                        "cudaMemsetAsync");
    if (rc) return rc;
    const int num_tiles = bins->tiles_x * bins->tiles_y;
    auto launch = [&](auto kernel) {
        kernel<<<num_tiles, kTilePixels, 0, stream>>>(
            splats, bins->sorted_idx, reinterpret_cast<const uint2 *>(bins->tile_ranges), bins->width,
            bins->height, bins->tiles_x, reinterpret_cast<const float4 *>(dl_dout), final_T,
            last_contrib, ctx->grad_acc);
    };
    if (ctx->opt_warp_skip && ctx->opt_last_contrib) launch(k_backward<true, true>);
    else if (ctx->opt_warp_skip) launch(k_backward<true, false>);
    else if (ctx->opt_last_contrib) launch(k_backward<false, true>);
    else launch(k_backward<false, false>);
    ++ctx->launches;
    if ((rc = cuda_check(ctx, cudaGetLastError(), "backward launch"))) return rc;
    const int blocks = (int)std::min<size_t>((count + 255) / 256, (size_t)SM_BLOCKS_CAP);
    k_grad_to_float<<<blocks, 256, 0, stream>>>(ctx->grad_acc, grad, count);
    ++ctx->launches;
    return cuda_check(ctx, cudaGetLastError(), "gradient conversion launch");
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
// name in host code is only a stand-in, not a device pointer).
double *g_noalloc_ptr[64] = {};

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
    double *acc = g_noalloc_ptr[ctx->device];
    if (!acc) {
        // First call on this device (the device is current here): find the
        // array's device address.
        void *p = nullptr;
        int rc = cuda_check(ctx, cudaGetSymbolAddress(&p, g_noalloc_grad_acc), "cudaGetSymbolAddress");
        if (rc) return rc;
        acc = static_cast<double *>(p);
        g_noalloc_ptr[ctx->device] = acc;
    }
    const size_t count = (size_t)n * 9;
    // The array keeps the previous call's sums: clear the part this call uses.
    int rc = cuda_check(ctx, cudaMemsetAsync(acc, 0, count * sizeof(double), stream), "cudaMemsetAsync");
    if (rc) return rc;
    const int num_tiles = bins->tiles_x * bins->tiles_y;
    auto launch = [&](auto kernel) {
        kernel<<<num_tiles, kTilePixels, 0, stream>>>(
            splats, bins->sorted_idx, reinterpret_cast<const uint2 *>(bins->tile_ranges), bins->width,
            bins->height, bins->tiles_x, reinterpret_cast<const float4 *>(dl_dout), final_T,
            last_contrib, acc);
    };
    if (ctx->opt_warp_skip && ctx->opt_last_contrib) launch(k_backward<true, true>);
    else if (ctx->opt_warp_skip) launch(k_backward<true, false>);
    else if (ctx->opt_last_contrib) launch(k_backward<false, true>);
    else launch(k_backward<false, false>);
    ++ctx->launches;
    if ((rc = cuda_check(ctx, cudaGetLastError(), "backward launch"))) return rc;
    const int blocks = (int)std::min<size_t>((count + 255) / 256, (size_t)SM_BLOCKS_CAP);
    k_grad_to_float<<<blocks, 256, 0, stream>>>(acc, grad, count);
    ++ctx->launches;
    return cuda_check(ctx, cudaGetLastError(), "gradient conversion launch");
}

}  // namespace gsr
