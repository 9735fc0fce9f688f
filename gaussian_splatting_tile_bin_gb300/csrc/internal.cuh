// internal.cuh -- definitions shared by the translation units of libgsr.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "gsr.h"

namespace gsr {

constexpr int kTile = GSR_TILE;           // 16x16 pixels per tile
constexpr int kTilePixels = kTile * kTile;
constexpr int kBinBlock = 256;            // splats per block in count / emit

// The three key/value buffers of a radix sort: buffer 0 holds the unsorted
// input, buffer 1 the sorted result, buffer 2 is ping-pong scratch.
template <typename K>
struct SortBuffers {
    K *k[3];
    uint32_t *v[3];
};
using PairBuffers = SortBuffers<uint64_t>;   // (tile << 32 | depth bits, splat index)
using DepthBuffers = SortBuffers<uint32_t>;  // (depth bits, splat index)

}  // namespace gsr

#include "context.h"

namespace gsr {

// Programmatic dependent launch.  Every kernel of the library starts with this:
// it lets the next grid in the stream begin launching (its CTAs take SM slots
// as this grid's CTAs retire), then waits until every grid before it in the
// stream has completed and its memory is visible.  No global memory is touched
// before the wait, so each kernel sees exactly what stream order promises.
__device__ __forceinline__ void grid_dependency_begin()
{
#if defined(__CUDA_ARCH__)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Race canary (a build with -DGSR_RACE_CANARY, for tests): at the call sites a
// warp sleeps a pseudo-random time that depends on its CTA, its warp and the
// site, so warps interleave differently from an unperturbed build.  A kernel
// whose results change under it depends on an ordering that no barrier or
// atomic guarantees.  In the normal build the sites compile to nothing.
#ifdef GSR_RACE_CANARY
__device__ __forceinline__ void race_canary(uint32_t site)
{
    uint32_t h = (blockIdx.x * 0x9E3779B1u) ^ ((threadIdx.x >> 5) * 0x85EBCA77u) ^ (site * 0xC2B2AE3Du);
    h ^= h >> 15;
    h *= 0x2C1B3C6Du;
    h ^= h >> 12;
    __nanosleep(h & 511u);
}
#define GSR_CANARY(site) ::gsr::race_canary(site)
#else
#define GSR_CANARY(site) ((void)0)
#endif

// Launches `kernel` on `stream`, with programmatic stream serialisation when the
// context allows it (GSR_OPT_PDL), and counts the launch.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(gsr_ctx *ctx, void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t stream,
                          Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = ctx->opt_pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ++ctx->launches;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// cudaMalloc for the context's arena and scratch.  With the context's test
// hook armed (GSR_OPT_FAIL_NEXT_ALLOC) it fails once, as an out-of-memory would.
inline cudaError_t device_alloc(gsr_ctx *ctx, void **ptr, size_t bytes)
{
    if (ctx->fail_next_alloc) {
        ctx->fail_next_alloc = 0;
        *ptr = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(ptr, bytes);
}

// Records a CUDA error on the context; returns GSR_ERR_CUDA (or GSR_OK).
int cuda_check(gsr_ctx *ctx, cudaError_t e, const char *what);
int fail(gsr_ctx *ctx, int code, const std::string &msg);

// Writes into order[0, num_tiles) every tile index once, tiles of larger cost
// first.  cost: the tile's list length from ranges (uint2 per tile) when
// ranges is set, else costs[tile].  Ties and near-ties (costs within one of 256
// logarithmic classes) come in any order.
int launch_tile_order(gsr_ctx *ctx, const uint32_t *ranges, const uint32_t *costs, int num_tiles, uint32_t *order,
                      cudaStream_t stream);

// Host sides of the three operations (validated arguments).
int bin_splats(gsr_ctx *ctx, const float *splats, const float *depths, int32_t n, int32_t width,
               int32_t height, cudaStream_t stream, gsr_bins *out);
int bin_pass_masks(gsr_ctx *ctx, uint32_t *depth_mask, uint32_t *tile_mask, int *tile_digit_bits,
                   int *tile_digits);
// The last binning's pair count, status (GSR_OK or GSR_ERR_TOO_MANY_PAIRS) and
// emitting splats, read from the device after waiting for its stream.
int bin_result(gsr_ctx *ctx, uint32_t *count, uint32_t *status, uint32_t *emitting);
int rasterize_forward(gsr_ctx *ctx, const float *splats, const gsr_bins *bins, float *out_rgbw,
                      float *final_T, uint32_t *last_contrib, cudaStream_t stream);
int rasterize_backward(gsr_ctx *ctx, const float *splats, int32_t n, const gsr_bins *bins,
                       const float *dl_dout, const float *final_T, const uint32_t *last_contrib,
                       float *grad, cudaStream_t stream);
int rasterize_backward_noalloc(gsr_ctx *ctx, const float *splats, int32_t n, const gsr_bins *bins,
                               const float *dl_dout, const float *final_T,
                               const uint32_t *last_contrib, float *grad, cudaStream_t stream);
int project_forward(gsr_ctx *ctx, const float *gauss, int32_t n, const gsr_camera &camera, float *splats,
                    float *depths, cudaStream_t stream);
int project_backward(gsr_ctx *ctx, const float *gauss, int32_t n, const gsr_camera &camera,
                     const float *dl_dsplat, float *dl_dg, cudaStream_t stream);
// out[i] = the raster kernels' exp(-s[i]).
int exp_neg_eval(gsr_ctx *ctx, const float *s, float *out, int32_t n, cudaStream_t stream);
// One launch of the FP32 / SFU rate kernel (peak.cu); *lane_ops = its lane operations.
int peak_kernel(gsr_ctx *ctx, int kind, int32_t iters, float *sink, uint64_t *lane_ops, cudaStream_t stream);

}  // namespace gsr
