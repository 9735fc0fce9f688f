// bin.cu -- tile binning: per-splat tile counts, a block scan, load-balanced
// pair emission, a stable LSD radix sort with 8-bit digits that skips every
// pass whose digit is the same in all keys, and per-tile range extraction.
//
// Follows "C0 resident arena + C1 pass skip" (p2-c0-resident-binning),
// section 2 table: key = (tile_id << 32) | depth_bits; a stable radix sort; a
// pass over a digit every key shares is the identity and is skipped (the page
// derives the skip from num_tiles for 4-bit digits; here the constant digits
// are found on the device from the AND and OR of all keys, which also catches
// constant depth-exponent digits); ranges extracted from the sorted keys; all
// buffers kept in a grow-only arena.
//
// The tile rectangle is computed with round-to-nearest intrinsics only (no
// contraction), so every splat's rectangle is the IEEE single-precision result
// of the same expression on any conforming implementation.
#include <algorithm>

#include "internal.cuh"

namespace gsr {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// The 3-sigma box of splat i as an inclusive tile rectangle (x0, y0, x1, y1).
// false when the splat is culled.
__device__ __forceinline__ bool splat_tile_rect(const float *__restrict__ splats,
                                                const float *__restrict__ depths, int i,
                                                int tiles_x, int tiles_y, int4 &r,
                                                uint32_t &depth_bits)
{
    const float *s = splats + 9 * (size_t)i;
    float v[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) v[k] = __ldg(s + k);
    float depth = __ldg(depths + i);
    bool ok = isfinite(depth) && depth > 0.0f;
#pragma unroll
    for (int k = 0; k < 9; ++k) ok = ok && isfinite(v[k]);
    if (!ok) return false;
    float a = v[2], b = v[3], c = v[4];
    float det = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, b));
    if (!(a > 0.0f) || !(det > 0.0f)) return false;
    float rx = __fmul_rn(3.0f, __fsqrt_rn(__fdiv_rn(c, det)));
    float ry = __fmul_rn(3.0f, __fsqrt_rn(__fdiv_rn(a, det)));
    float fx0 = __fmul_rn(__fsub_rn(v[0], rx), 0.0625f);
    float fx1 = __fmul_rn(__fadd_rn(v[0], rx), 0.0625f);
    float fy0 = __fmul_rn(__fsub_rn(v[1], ry), 0.0625f);
    float fy1 = __fmul_rn(__fadd_rn(v[1], ry), 0.0625f);
    const float mx = (float)tiles_x, my = (float)tiles_y;
    int x0 = (int)floorf(fminf(fmaxf(fx0, -1.0f), mx));
    int x1 = (int)floorf(fminf(fmaxf(fx1, -1.0f), mx));
    int y0 = (int)floorf(fminf(fmaxf(fy0, -1.0f), my));
    int y1 = (int)floorf(fminf(fmaxf(fy1, -1.0f), my));
    x0 = max(x0, 0);
    y0 = max(y0, 0);
    x1 = min(x1, tiles_x - 1);
    y1 = min(y1, tiles_y - 1);
    if (x0 > x1 || y0 > y1) return false;
    r = make_int4(x0, y0, x1, y1);
    depth_bits = __float_as_uint(depth);
    return true;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Exclusive scan over a 256-thread block; returns the exclusive prefix and the
// block total in *total.  `ws` must hold 8 elements.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan_256(T v, T *ws, T *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    T warp_off = 0, sum = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        T x = ws[w];
        if (w < warp) warp_off += x;
        sum += x;
    }
    __syncthreads();
    *total = sum;
    return warp_off + incl - v;
}

// --- count -----------------------------------------------------------------

__global__ void __launch_bounds__(kBinBlock)
k_count(const float *__restrict__ splats, const float *__restrict__ depths, int n, int tiles_x,
        int tiles_y, uint32_t *__restrict__ counts, unsigned long long *__restrict__ blk_sums)
{
    const int i = blockIdx.x * kBinBlock + threadIdx.x;
    uint32_t c = 0;
    if (i < n) {
        int4 r;
        uint32_t db;
        if (splat_tile_rect(splats, depths, i, tiles_x, tiles_y, r, db))
            c = (uint32_t)(r.z - r.x + 1) * (uint32_t)(r.w - r.y + 1);
        counts[i] = c;
    }
    __shared__ unsigned long long ws[8];
    unsigned long long v = warp_sum<unsigned long long>(c);
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < 8; ++w) t += ws[w];
        blk_sums[blockIdx.x] = t;
    }
}

// One block: exclusive scan of the per-block sums, the pair total, and the
// AND/OR accumulators reset for the emission.
__global__ void __launch_bounds__(1024)
k_scan_blocks(const unsigned long long *__restrict__ blk_sums, int nblk,
              unsigned long long *__restrict__ blk_offs, unsigned long long *__restrict__ scalars)
{
    __shared__ unsigned long long ws[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long carry = 0;
    for (int base = 0; base < nblk; base += 1024) {
        const int i = base + threadIdx.x;
        unsigned long long v = i < nblk ? blk_sums[i] : 0ull;
        unsigned long long incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned long long x = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) ws[warp] = incl;
        __syncthreads();
        unsigned long long off = 0, sum = 0;
        for (int w = 0; w < 32; ++w) {
            if (w < warp) off += ws[w];
            sum += ws[w];
        }
        __syncthreads();
        if (i < nblk) blk_offs[i] = carry + off + incl - v;
        carry += sum;
    }
    if (threadIdx.x == 0) {
        scalars[0] = carry;
        scalars[1] = ~0ull;
        scalars[2] = 0ull;
    }
}

// --- emit ------------------------------------------------------------------

// Each block re-derives the rectangles of its 256 splats, scans their counts
// and writes its contiguous slice of pairs with all 256 threads, so a splat
// with thousands of tiles does not serialise on one thread.  Within a splat the
// pairs go in row-major tile order; across splats in splat order.
__global__ void __launch_bounds__(kBinBlock)
k_emit(const float *__restrict__ splats, const float *__restrict__ depths, int n, int tiles_x,
       int tiles_y, const unsigned long long *__restrict__ blk_offs, uint64_t *__restrict__ keys,
       uint32_t *__restrict__ vals, unsigned long long *__restrict__ scalars)
{
    __shared__ uint32_t s_off[kBinBlock];
    __shared__ int4 s_rect[kBinBlock];
    __shared__ uint32_t s_db[kBinBlock];
    __shared__ uint32_t ws[8];
    __shared__ unsigned long long s_and[8], s_or[8];

    const int i = blockIdx.x * kBinBlock + threadIdx.x;
    uint32_t c = 0;
    int4 r = make_int4(0, 0, -1, -1);
    uint32_t db = 0;
    if (i < n && splat_tile_rect(splats, depths, i, tiles_x, tiles_y, r, db))
        c = (uint32_t)(r.z - r.x + 1) * (uint32_t)(r.w - r.y + 1);
    uint32_t total;
    const uint32_t excl = block_exclusive_scan_256<uint32_t>(c, ws, &total);
    s_off[threadIdx.x] = excl;
    s_rect[threadIdx.x] = r;
    s_db[threadIdx.x] = db;
    __syncthreads();

    const unsigned long long base = blk_offs[blockIdx.x];
    unsigned long long acc_and = ~0ull, acc_or = 0ull;
    for (uint32_t q = threadIdx.x; q < total; q += kBinBlock) {
        // Last splat t with s_off[t] <= q; it has a nonzero count.
        int lo = 0, hi = kBinBlock - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= q) lo = mid;
            else hi = mid - 1;
        }
        const int4 rr = s_rect[lo];
        const uint32_t local = q - s_off[lo];
        const uint32_t w = (uint32_t)(rr.z - rr.x + 1);
        const uint32_t dy = local / w;
        const uint32_t ty = (uint32_t)rr.y + dy;
        const uint32_t tx = (uint32_t)rr.x + (local - dy * w);
        const uint64_t tile = (uint64_t)ty * (uint64_t)tiles_x + tx;
        const uint64_t key = (tile << 32) | (uint64_t)s_db[lo];
        keys[base + q] = key;
        vals[base + q] = (uint32_t)(blockIdx.x * kBinBlock + lo);
        acc_and &= key;
        acc_or |= key;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc_and &= __shfl_xor_sync(kFull, acc_and, o);
        acc_or |= __shfl_xor_sync(kFull, acc_or, o);
    }
    if ((threadIdx.x & 31) == 0) {
        s_and[threadIdx.x >> 5] = acc_and;
        s_or[threadIdx.x >> 5] = acc_or;
    }
    __syncthreads();
    if (threadIdx.x == 0 && total > 0) {
        unsigned long long a = ~0ull, o = 0ull;
        for (int w = 0; w < 8; ++w) {
            a &= s_and[w];
            o |= s_or[w];
        }
        atomicAnd(&scalars[1], a);
        atomicOr(&scalars[2], o);
    }
}

// --- radix sort --------------------------------------------------------------

// Buffer b of the three (a select, so the kernel parameter block is not copied
// to local memory for dynamic indexing).
__device__ __forceinline__ uint64_t *keys_of(const PairBuffers &p, int b)
{
    return b == 0 ? p.k[0] : (b == 1 ? p.k[1] : p.k[2]);
}
__device__ __forceinline__ uint32_t *vals_of(const PairBuffers &p, int b)
{
    return b == 0 ? p.v[0] : (b == 1 ? p.v[1] : p.v[2]);
}

// Decides which 8-bit digits vary and chains the executed passes so that the
// last one writes buffer 1: pass j of k reads the previous pass's output (the
// emitted buffer 0 for the first) and writes buffer 1 when k - 1 - j is even,
// buffer 2 otherwise.
__global__ void k_radix_plan(const unsigned long long *__restrict__ scalars, int digits,
                             RadixPlan *__restrict__ plan)
{
    if (threadIdx.x != 0) return;
    const unsigned long long diff = scalars[1] ^ scalars[2];
    int list[kMaxDigits];
    int k = 0;
    for (int d = 0; d < kMaxDigits; ++d) {
        const bool ex = d < digits && ((diff >> (8 * d)) & 0xffull) != 0ull;
        plan->exec[d] = ex ? 1 : 0;
        plan->src[d] = 0;
        plan->dst[d] = 0;
        if (ex) list[k++] = d;
    }
    int prev = 0;
    for (int j = 0; j < k; ++j) {
        const int d = list[j];
        const int dst = ((k - 1 - j) % 2 == 0) ? 1 : 2;
        plan->src[d] = prev;
        plan->dst[d] = dst;
        prev = dst;
    }
    plan->num_exec = k;
}

// Per radix tile: how many keys carry each digit value.  counts is
// digit-major, [256][ntiles]; totals[digit] accumulates over tiles.
__global__ void __launch_bounds__(kRadixThreads)
k_radix_upsweep(const RadixPlan *__restrict__ plan, int d, PairBuffers bufs, uint32_t num,
                int ntiles, uint32_t *__restrict__ counts, uint32_t *__restrict__ totals)
{
    if (!plan->exec[d]) return;
    const uint64_t *__restrict__ keys = keys_of(bufs, plan->src[d]);
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const int shift = 8 * d;
    const uint32_t base = blockIdx.x * kRadixTile;
#pragma unroll
    for (int k = 0; k < kRadixItems; ++k) {
        const uint32_t i = base + k * kRadixThreads + threadIdx.x;
        if (i < num) atomicAdd(&h[(uint32_t)(keys[i] >> shift) & 0xffu], 1u);
    }
    __syncthreads();
    const uint32_t c = h[threadIdx.x];
    counts[(size_t)threadIdx.x * ntiles + blockIdx.x] = c;
    if (c) atomicAdd(&totals[threadIdx.x], c);
}

// One block per digit value: the global start of the digit (sum of the totals
// of smaller digits) plus an exclusive scan of that digit's per-tile counts,
// written in place.
__global__ void __launch_bounds__(kRadixThreads)
k_radix_scan(const RadixPlan *__restrict__ plan, int d, int ntiles, uint32_t *__restrict__ counts,
             const uint32_t *__restrict__ totals)
{
    if (!plan->exec[d]) return;
    __shared__ uint32_t ws[8];
    const uint32_t digit = blockIdx.x;
    uint32_t dummy, base;
    {
        const uint32_t x = threadIdx.x < digit ? totals[threadIdx.x] : 0u;
        block_exclusive_scan_256<uint32_t>(x, ws, &base);
    }
    uint32_t *row = counts + (size_t)digit * ntiles;
    uint32_t carry = base;
    for (int start = 0; start < ntiles; start += kRadixThreads) {
        const int i = start + threadIdx.x;
        const uint32_t c = i < ntiles ? row[i] : 0u;
        uint32_t sum;
        const uint32_t e = block_exclusive_scan_256<uint32_t>(c, ws, &sum);
        if (i < ntiles) row[i] = carry + e;
        carry += sum;
    }
    (void)dummy;
}

// Stable scatter of one radix tile.  Warp w owns keys [w*256, w*256+256) of
// the tile and walks them in 8 rounds of 32 consecutive keys; within a round
// equal digits are ranked by lane (match.any), across rounds by per-warp digit
// counters, across warps by a per-digit prefix over the 8 warps, across tiles
// by the scanned counts.  This reproduces input order among equal digits.
__global__ void __launch_bounds__(kRadixThreads)
k_radix_downsweep(const RadixPlan *__restrict__ plan, int d, PairBuffers bufs, uint32_t num,
                  int ntiles, const uint32_t *__restrict__ offsets)
{
    if (!plan->exec[d]) return;
    const int src = plan->src[d], dst = plan->dst[d];
    const uint64_t *__restrict__ kin = keys_of(bufs, src);
    const uint32_t *__restrict__ vin = vals_of(bufs, src);
    uint64_t *__restrict__ kout = keys_of(bufs, dst);
    uint32_t *__restrict__ vout = vals_of(bufs, dst);

    __shared__ uint32_t wcnt[8][256];
    __shared__ uint32_t toff[256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int k = threadIdx.x; k < 8 * 256; k += kRadixThreads) (&wcnt[0][0])[k] = 0;
    toff[threadIdx.x] = offsets[(size_t)threadIdx.x * ntiles + blockIdx.x];
    __syncthreads();

    const int shift = 8 * d;
    const uint32_t lanemask_lt = (1u << lane) - 1u;
    const uint32_t base = blockIdx.x * kRadixTile + warp * (32 * kRadixItems);
    uint64_t key[kRadixItems];
    uint32_t val[kRadixItems];
    uint32_t rank[kRadixItems];
#pragma unroll
    for (int k = 0; k < kRadixItems; ++k) {
        const uint32_t i = base + k * 32 + lane;
        const bool valid = i < num;
        key[k] = valid ? kin[i] : 0ull;
        val[k] = valid ? vin[i] : 0u;
        const uint32_t digit = valid ? ((uint32_t)(key[k] >> shift) & 0xffu) : 0x100u;
        const uint32_t peers = __match_any_sync(kFull, digit);
        const uint32_t prior = valid ? wcnt[warp][digit] : 0u;
        __syncwarp();
        const uint32_t before = __popc(peers & lanemask_lt);
        if (valid && before == 0) wcnt[warp][digit] = prior + __popc(peers);
        __syncwarp();
        rank[k] = prior + before;
    }
    __syncthreads();
    {
        const int v = threadIdx.x;
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t t = wcnt[w][v];
            wcnt[w][v] = run;
            run += t;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRadixItems; ++k) {
        const uint32_t i = base + k * 32 + lane;
        if (i < num) {
            const uint32_t digit = (uint32_t)(key[k] >> shift) & 0xffu;
            const uint32_t pos = toff[digit] + wcnt[warp][digit] + rank[k];
            kout[pos] = key[k];
            vout[pos] = val[k];
        }
    }
}

// When every digit was constant no pass ran and the emitted order is already
// sorted; copy it to the result buffer.
__global__ void k_copy_if_unsorted(const RadixPlan *__restrict__ plan, PairBuffers bufs,
                                   uint32_t num)
{
    if (plan->num_exec != 0) return;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < num; i += gridDim.x * blockDim.x) {
        bufs.k[1][i] = bufs.k[0][i];
        bufs.v[1][i] = bufs.v[0][i];
    }
}

// --- ranges --------------------------------------------------------------------

__global__ void k_extract_ranges(const uint64_t *__restrict__ keys, uint32_t num,
                                 uint32_t *__restrict__ ranges)
{
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= num) return;
    const uint32_t t = (uint32_t)(keys[i] >> 32);
    if (i == 0 || (uint32_t)(keys[i - 1] >> 32) != t) ranges[2 * (size_t)t] = i;
    if (i == num - 1 || (uint32_t)(keys[i + 1] >> 32) != t) ranges[2 * (size_t)t + 1] = i + 1;
}

int bits_for(uint64_t v)
{
    int b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

template <typename T>
int grow(gsr_ctx *ctx, T **ptr, size_t *cap, size_t need, size_t elems_per, const char *what)
{
    if (need <= *cap && *ptr) return GSR_OK;
    if (*ptr) {
        cudaFree(*ptr);
        *ptr = nullptr;
    }
    *cap = 0;
    cudaError_t e = cudaMalloc((void **)ptr, std::max<size_t>(need, 1) * elems_per * sizeof(T));
    if (e != cudaSuccess) {
        cudaGetLastError();
        *ptr = nullptr;
        return fail(ctx, GSR_ERR_OOM, std::string("cudaMalloc failed for ") + what);
    }
    *cap = need;
    return GSR_OK;
}

}  // namespace

#define GSR_LAUNCHED(ctx)                                                     \
    do {                                                                      \
        ++(ctx)->launches;                                                    \
        int _rc = cuda_check((ctx), cudaGetLastError(), "kernel launch");     \
        if (_rc) return _rc;                                                  \
    } while (0)

int bin_splats(gsr_ctx *ctx, const float *splats, const float *depths, int32_t n, int32_t width,
               int32_t height, cudaStream_t stream, gsr_bins *out)
{
    int rc;
    const int tiles_x = (width + kTile - 1) / kTile;
    const int tiles_y = (height + kTile - 1) / kTile;
    const size_t num_tiles = (size_t)tiles_x * tiles_y;
    const int key_bits = 32 + bits_for(num_tiles - 1);
    const int digits = (key_bits + 7) / 8;

    // Fixed-size scratch, allocated once.
    if (!ctx->scalars) {
        if ((rc = cuda_check(ctx, cudaMalloc(&ctx->scalars, 4 * sizeof(unsigned long long)), "cudaMalloc")))
            return rc;
        if ((rc = cuda_check(ctx, cudaMalloc(&ctx->radix_totals, kMaxDigits * 256 * sizeof(uint32_t)),
                             "cudaMalloc")))
            return rc;
        if ((rc = cuda_check(ctx, cudaMalloc(&ctx->plan, sizeof(RadixPlan)), "cudaMalloc"))) return rc;
        if ((rc = cuda_check(ctx, cudaHostAlloc(&ctx->host_total, sizeof(unsigned long long),
                                                cudaHostAllocDefault),
                             "cudaHostAlloc")))
            return rc;
    }
    const int nblk = (n + kBinBlock - 1) / kBinBlock;
    if ((rc = grow(ctx, &ctx->counts, &ctx->cap_splats, (size_t)n, 1, "counts"))) return rc;
    // Block sums and block offsets share one buffer: [0, cap) and [cap, 2 cap).
    if ((rc = grow(ctx, &ctx->blk_sums, &ctx->cap_blocks, (size_t)nblk, 2, "block sums"))) return rc;
    ctx->blk_offs = ctx->blk_sums + ctx->cap_blocks;
    if ((rc = grow(ctx, &ctx->ranges, &ctx->cap_tiles, num_tiles, 2, "tile ranges"))) return rc;

    // 1. count + scan, then read the pair total.
    uint64_t total = 0;
    if (n > 0) {
        k_count<<<nblk, kBinBlock, 0, stream>>>(splats, depths, n, tiles_x, tiles_y, ctx->counts,
                                                ctx->blk_sums);
        GSR_LAUNCHED(ctx);
        k_scan_blocks<<<1, 1024, 0, stream>>>(ctx->blk_sums, nblk, ctx->blk_offs, ctx->scalars);
        GSR_LAUNCHED(ctx);
        if ((rc = cuda_check(ctx, cudaMemcpyAsync(ctx->host_total, ctx->scalars, sizeof(unsigned long long),
                                                  cudaMemcpyDeviceToHost, stream),
                             "cudaMemcpyAsync")))
            return rc;
        if ((rc = cuda_check(ctx, cudaStreamSynchronize(stream), "cudaStreamSynchronize"))) return rc;
        total = *ctx->host_total;
    }
    if (total > (uint64_t)GSR_MAX_PAIRS)
        return fail(ctx, GSR_ERR_TOO_MANY_PAIRS,
                    "tile-pair count " + std::to_string(total) + " exceeds GSR_MAX_PAIRS");
    const uint32_t num = (uint32_t)total;

    // 2. grow the pair buffers: max(65536, 16 n, 1.5 x pairs).
    if (num > ctx->cap_pairs || !ctx->pairs.k[0]) {
        size_t cap = std::max<size_t>(65536, (size_t)16 * (size_t)n);
        cap = std::max<size_t>(cap, (size_t)num + num / 2);
        cap = std::min<size_t>(cap, (size_t)GSR_MAX_PAIRS);
        cap = std::max<size_t>(cap, num);
        for (int b = 0; b < 3; ++b) {
            if (ctx->pairs.k[b]) cudaFree(ctx->pairs.k[b]);
            if (ctx->pairs.v[b]) cudaFree(ctx->pairs.v[b]);
            ctx->pairs.k[b] = nullptr;
            ctx->pairs.v[b] = nullptr;
        }
        ctx->cap_pairs = 0;
        for (int b = 0; b < 3; ++b) {
            if (cudaMalloc(&ctx->pairs.k[b], cap * sizeof(uint64_t)) != cudaSuccess ||
                cudaMalloc(&ctx->pairs.v[b], cap * sizeof(uint32_t)) != cudaSuccess) {
                cudaGetLastError();
                return fail(ctx, GSR_ERR_OOM,
                            "cudaMalloc failed for " + std::to_string(cap) + " tile pairs");
            }
        }
        ctx->cap_pairs = cap;
    }
    const int ntiles = (int)((num + kRadixTile - 1) / kRadixTile);
    if ((rc = grow(ctx, &ctx->radix_counts, &ctx->cap_radix_tiles, (size_t)std::max(ntiles, 1), 256,
                   "radix counts")))
        return rc;

    if ((rc = cuda_check(ctx, cudaMemsetAsync(ctx->ranges, 0, num_tiles * 2 * sizeof(uint32_t), stream),
                         "cudaMemsetAsync")))
        return rc;

    if (num > 0) {
        // 3. emission.
        k_emit<<<nblk, kBinBlock, 0, stream>>>(splats, depths, n, tiles_x, tiles_y, ctx->blk_offs,
                                               ctx->pairs.k[0], ctx->pairs.v[0], ctx->scalars);
        GSR_LAUNCHED(ctx);
        // 4. radix sort over the digits the keys can occupy; constant ones skip on the device.
        k_radix_plan<<<1, 32, 0, stream>>>(ctx->scalars, digits, ctx->plan);
        GSR_LAUNCHED(ctx);
        if ((rc = cuda_check(ctx, cudaMemsetAsync(ctx->radix_totals, 0,
                                                  kMaxDigits * 256 * sizeof(uint32_t), stream),
                             "cudaMemsetAsync")))
            return rc;
        for (int d = 0; d < digits; ++d) {
            uint32_t *totals = ctx->radix_totals + 256 * d;
            k_radix_upsweep<<<ntiles, kRadixThreads, 0, stream>>>(ctx->plan, d, ctx->pairs, num, ntiles,
                                                                  ctx->radix_counts, totals);
            GSR_LAUNCHED(ctx);
            k_radix_scan<<<256, kRadixThreads, 0, stream>>>(ctx->plan, d, ntiles, ctx->radix_counts,
                                                            totals);
            GSR_LAUNCHED(ctx);
            k_radix_downsweep<<<ntiles, kRadixThreads, 0, stream>>>(ctx->plan, d, ctx->pairs, num,
                                                                    ntiles, ctx->radix_counts);
            GSR_LAUNCHED(ctx);
        }
        k_copy_if_unsorted<<<std::min(ntiles, 1024), 256, 0, stream>>>(ctx->plan, ctx->pairs, num);
        GSR_LAUNCHED(ctx);
        // 5. per-tile ranges.
        k_extract_ranges<<<(num + 255) / 256, 256, 0, stream>>>(ctx->pairs.k[1], num, ctx->ranges);
        GSR_LAUNCHED(ctx);
    }

    ctx->last_stream = stream;
    ctx->last_pairs = num;
    ctx->last_key_digits = digits;
    out->keys = ctx->pairs.k[1];
    out->sorted_idx = ctx->pairs.v[1];
    out->tile_ranges = ctx->ranges;
    out->num_pairs = num;
    out->n = n;
    out->width = width;
    out->height = height;
    out->tiles_x = tiles_x;
    out->tiles_y = tiles_y;
    return GSR_OK;
}

}  // namespace gsr
