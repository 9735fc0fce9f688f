// bin.cu -- tile binning.
//
// Follows "C0 resident arena + C1 pass skip" (p2-c0-resident-binning),
// section 2 table: each splat emits a key (tile_id << 32) | depth_bits per tile
// it touches, the pairs are sorted by key with a stable radix sort whose passes
// over constant digits are skipped, per-tile ranges are extracted from the
// sorted keys, and every buffer lives in a grow-only arena.
//
// The sorted order is (tile, depth bits, splat index).  It is produced in two
// stages that give exactly the same keys and indices as sorting the pairs on
// the whole key:
//   1. the splats that emit at least one pair are compacted and sorted stably
//      by their depth bits (LSD, 8-bit digits, 4 passes at most over the
//      splats instead of over the pairs);
//   2. the pairs are emitted in that depth order (a splat's own pairs in
//      row-major tile order), so they are already ordered by (depth, index)
//      within every tile, and a stable LSD sort on the tile digits alone
//      finishes the job.  The tile field is split into digits of equal width
//      (two 6-bit digits for 2500 tiles), which keeps the buckets few and the
//      scattered runs long.
// In both sorts a digit that every key shares is found on the device from the
// AND and the OR of all keys, and its pass is skipped.
//
// The tile rectangle is computed with round-to-nearest intrinsics only (no
// contraction), so every splat's rectangle is the IEEE single-precision result
// of the same expression on any conforming implementation.
#include <algorithm>

#include "internal.cuh"

namespace gsr {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ctx->scalars slots.
enum {
    kScalarPairs = 0,      // total tile pairs
    kScalarEmitting = 1,   // splats with at least one pair
    kScalarDepthAnd = 2,   // AND / OR of the emitting splats' depth bits
    kScalarDepthOr = 3,
    kScalarKeyAnd = 4,     // AND / OR of the emitted keys
    kScalarKeyOr = 5,
    kScalarTicketCount = 6,  // blocks of k_count / k_sorted_sums done (the last one scans)
    kScalarTicketSums = 7,
    kScalarNum = 8,        // pairs the sort and the ranges take: the total, or 0 when it exceeds the capacity
    kScalarResult = 9,     // two uint32: the pair count (saturated) and the status (GSR_OK or
                           // GSR_ERR_TOO_MANY_PAIRS); gsr_bins.num_pairs_dev points here
    kScalarCount = 10
};

// The 3-sigma box of a splat (its 9 fields v and its depth) as an inclusive
// tile rectangle (x0, y0, x1, y1).  false when the splat is culled.
__device__ __forceinline__ bool tile_rect(const float (&v)[9], float depth, int tiles_x, int tiles_y, int4 &r)
{
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
    return true;
}

// A tile rectangle packed into 8 bytes: (x0 | y0 << 16, x1 | y1 << 16); tile
// coordinates fit 16 bits (at most 32768 tiles per side).  A culled splat is
// stored as x0 = 1 > x1 = 0.
__device__ __forceinline__ uint2 pack_rect(bool ok, int4 r)
{
    return ok ? make_uint2((uint32_t)r.x | ((uint32_t)r.y << 16), (uint32_t)r.z | ((uint32_t)r.w << 16))
              : make_uint2(1u, 0u);
}

__device__ __forceinline__ uint32_t rect_width(uint2 p) { return (p.y & 0xffffu) - (p.x & 0xffffu) + 1u; }
__device__ __forceinline__ uint32_t rect_count(uint2 p)
{
    const uint32_t x0 = p.x & 0xffffu, x1 = p.y & 0xffffu, y0 = p.x >> 16, y1 = p.y >> 16;
    return x0 <= x1 && y0 <= y1 ? (x1 - x0 + 1u) * (y1 - y0 + 1u) : 0u;
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

// AND and OR of one value per thread over a 256-thread block, folded into
// acc[0] (AND) and acc[1] (OR) by thread 0.  Threads pass ~0 / 0 to abstain.
__device__ __forceinline__ void block_and_or_into(unsigned long long a, unsigned long long o,
                                                  unsigned long long *s_and, unsigned long long *s_or,
                                                  unsigned long long *acc)
{
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) {
        a &= __shfl_xor_sync(kFull, a, k);
        o |= __shfl_xor_sync(kFull, o, k);
    }
    if ((threadIdx.x & 31) == 0) {
        s_and[threadIdx.x >> 5] = a;
        s_or[threadIdx.x >> 5] = o;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long ta = ~0ull, to = 0ull;
        for (int w = 0; w < 8; ++w) {
            ta &= s_and[w];
            to |= s_or[w];
        }
        if (ta != ~0ull) atomicAnd(acc, ta);
        if (to != 0ull) atomicOr(acc + 1, to);
    }
}

// The block's AND / OR of (a, o), valid in thread 0.
__device__ __forceinline__ void block_and_or(unsigned long long &a, unsigned long long &o, unsigned long long *s_and,
                                             unsigned long long *s_or)
{
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) {
        a &= __shfl_xor_sync(kFull, a, k);
        o |= __shfl_xor_sync(kFull, o, k);
    }
    if ((threadIdx.x & 31) == 0) {
        s_and[threadIdx.x >> 5] = a;
        s_or[threadIdx.x >> 5] = o;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 8; ++w) {
            a &= s_and[w];
            o |= s_or[w];
        }
    }
    __syncthreads();
}

// Lanes in `members` whose kWidth-bit digit equals this lane's, from one
// ballot per bit.  Every lane of the warp calls this together.
template <int kWidth>
__device__ __forceinline__ uint32_t digit_peers(uint32_t members, uint32_t digit)
{
    uint32_t peers = members;
#pragma unroll
    for (int b = 0; b < kWidth; ++b) {
        const uint32_t bal = __ballot_sync(kFull, (digit >> b) & 1u);
        peers &= ((digit >> b) & 1u) ? bal : ~bal;
    }
    return peers;
}

// Radix digits: the key bits [key_lo, key_hi) split into num_fields digits of
// equal width, at most 8 bits each.
__host__ __device__ __forceinline__ int num_fields(int key_lo, int key_hi)
{
    return (key_hi - key_lo + 7) / 8;
}

__host__ __device__ __forceinline__ void field_geom(int key_lo, int key_hi, int nfields, int f, int &shift,
                                                    int &width)
{
    const int w = (key_hi - key_lo + nfields - 1) / nfields;
    shift = key_lo + f * w;
    width = key_hi - shift < w ? key_hi - shift : w;
}

// Digit f of the keys varies iff its bits differ between the AND and the OR of
// all keys.
__host__ __device__ __forceinline__ bool field_varies(unsigned long long and_or_diff, int shift, int width)
{
    return width > 0 && ((and_or_diff >> shift) & ((1ull << width) - 1ull)) != 0ull;
}

// Position of `field` among the executed passes (-1 if skipped); *executed
// receives their number.  The executed passes chain buffer 0 -> ... -> 1:
// pass j of k writes buffer 1 when k - 1 - j is even, buffer 2 otherwise, and
// reads what pass j - 1 wrote (buffer 0 for the first).
__host__ __device__ __forceinline__ int field_pass(unsigned long long diff, int key_lo, int key_hi, int field,
                                                  int *executed)
{
    const int nf = num_fields(key_lo, key_hi);
    int k = 0, j = -1;
    for (int f = 0; f < nf; ++f) {
        int sh, w;
        field_geom(key_lo, key_hi, nf, f, sh, w);
        if (field_varies(diff, sh, w)) {
            if (f == field) j = k;
            ++k;
        }
    }
    *executed = k;
    return j;
}

// Clears the binning's scalars and the radix digit totals of both sorts.

// True in the one block that finishes last: every block calls this after it has
// written its per-block results, and the last block then reads all of them
// (the fences order each block's writes before its ticket).
__device__ __forceinline__ bool last_block_done(unsigned long long *ticket)
{
    __shared__ bool s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(ticket, 1ull) == (unsigned long long)(gridDim.x - 1);
    }
    __syncthreads();
    if (s_last) __threadfence();
    return s_last;
}

// Exclusive scan in place of vals[0, num) by one 256-thread block (reads that
// bypass L1: other blocks wrote the values); returns the total.  Each thread
// takes a contiguous run of the values: one block-wide scan of the runs' sums.
__device__ unsigned long long block_scan_inplace_256(unsigned long long *__restrict__ vals, int num,
                                                     unsigned long long *ws)
{
    const int per = (num + kBinBlock - 1) / kBinBlock;
    const int b0 = min(num, (int)threadIdx.x * per), b1 = min(num, b0 + per);
    unsigned long long sum = 0;
    for (int i = b0; i < b1; ++i) sum += __ldcg(vals + i);
    unsigned long long total;
    unsigned long long run = block_exclusive_scan_256<unsigned long long>(sum, ws, &total);
    for (int i = b0; i < b1; ++i) {
        const unsigned long long v = __ldcg(vals + i);
        vals[i] = run;
        run += v;
    }
    return total;
}

// --- count -----------------------------------------------------------------

// Per splat: its tile rectangle.  Per block: the pair total, the number of
// emitting splats, and the AND / OR of their depth bits.  The block's 256
// records (9216 contiguous bytes) are read with coalesced 4-byte loads through
// shared memory.
__global__ void __launch_bounds__(kBinBlock)
k_count(const float *__restrict__ splats, const float *__restrict__ depths, int n, int tiles_x,
        int tiles_y, uint2 *__restrict__ rects, unsigned long long *__restrict__ blk_pairs,
        unsigned long long *__restrict__ blk_emitting, unsigned long long *__restrict__ blk_and,
        unsigned long long *__restrict__ blk_or, unsigned long long *__restrict__ scalars,
        uint32_t *__restrict__ radix_totals, int ntotals, unsigned long long capacity)
{
    grid_dependency_begin();
    // Block 0 clears what the binning's later kernels accumulate into.
    if (blockIdx.x == 0) {
        for (int k = threadIdx.x; k < ntotals; k += kBinBlock) radix_totals[k] = 0u;
        if (threadIdx.x == 0) {
            scalars[kScalarTicketSums] = 0ull;
            scalars[kScalarKeyAnd] = ~0ull;
            scalars[kScalarKeyOr] = 0ull;
        }
    }
    __shared__ float s_rec[kBinBlock * 9];
    __shared__ unsigned long long s_and[8], s_or[8];
    __shared__ unsigned long long ws[8];
    const int first = blockIdx.x * kBinBlock;
    const int nrec = min(kBinBlock, n - first);
    const float *src = splats + 9 * (size_t)first;
#pragma unroll
    for (int k = 0; k < 9; ++k) {
        const int e = k * kBinBlock + threadIdx.x;
        if (e < nrec * 9) s_rec[e] = __ldg(src + e);
    }
    __syncthreads();
    const int i = first + threadIdx.x;
    uint32_t c = 0, db = 0;
    if (i < n) {
        float v[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) v[k] = s_rec[9 * threadIdx.x + k];
        const float depth = __ldg(depths + i);
        int4 r = make_int4(0, 0, 0, 0);
        const bool ok = tile_rect(v, depth, tiles_x, tiles_y, r);
        const uint2 pr = pack_rect(ok, r);
        rects[i] = pr;
        c = rect_count(pr);
        db = __float_as_uint(depth);
    }
    unsigned long long pairs_total, emit_total;
    block_exclusive_scan_256<unsigned long long>(c, ws, &pairs_total);
    block_exclusive_scan_256<unsigned long long>(c > 0 ? 1ull : 0ull, ws, &emit_total);
    if (threadIdx.x == 0) {
        blk_pairs[blockIdx.x] = pairs_total;
        blk_emitting[blockIdx.x] = emit_total;
    }
    unsigned long long da = c > 0 ? (unsigned long long)db : ~0ull, dor = c > 0 ? (unsigned long long)db : 0ull;
    block_and_or(da, dor, s_and, s_or);
    if (threadIdx.x == 0) {
        blk_and[blockIdx.x] = da;
        blk_or[blockIdx.x] = dor;
    }
    // The last block: the pair total (a plain sum), the exclusive scan of the
    // per-block emitting counts with their total, and the depth bits' AND / OR.
    if (last_block_done(scalars + kScalarTicketCount)) {
        unsigned long long s = 0, a = ~0ull, o = 0ull;
        for (int b = threadIdx.x; b < (int)gridDim.x; b += kBinBlock) {
            s += __ldcg(blk_pairs + b);
            a &= __ldcg(blk_and + b);
            o |= __ldcg(blk_or + b);
        }
        unsigned long long t;
        block_exclusive_scan_256<unsigned long long>(s, ws, &t);
        __syncthreads();
        block_and_or(a, o, s_and, s_or);
        const unsigned long long m = block_scan_inplace_256(blk_emitting, (int)gridDim.x, ws);
        if (threadIdx.x == 0) {
            scalars[kScalarDepthAnd] = a;
            scalars[kScalarDepthOr] = o;
            scalars[kScalarTicketCount] = 0ull;   // for the next binning
            // More pairs than the arena holds (or than 32-bit indices reach):
            // nothing is emitted, sorted or ranged, and every tile stays empty.
            const bool fits = t <= capacity && t <= (unsigned long long)GSR_MAX_PAIRS;
            scalars[kScalarPairs] = t;
            scalars[kScalarEmitting] = fits ? m : 0ull;
            scalars[kScalarNum] = fits ? t : 0ull;
            uint32_t *res = reinterpret_cast<uint32_t *>(scalars + kScalarResult);
            res[0] = t < 0xffffffffull ? (uint32_t)t : 0xffffffffu;
            res[1] = fits ? (uint32_t)GSR_OK : (uint32_t)GSR_ERR_TOO_MANY_PAIRS;
        }
    }
}

// Writes (depth bits, splat index) of every emitting splat, in splat order.
__global__ void __launch_bounds__(kBinBlock)
k_compact(const uint2 *__restrict__ rects, const float *__restrict__ depths, int n,
          const unsigned long long *__restrict__ blk_emit_offs, uint32_t *__restrict__ dkeys,
          uint32_t *__restrict__ didx, uint32_t *__restrict__ ranges, uint32_t range_words)
{
    grid_dependency_begin();
    __shared__ uint32_t ws[8];
    const int i = blockIdx.x * kBinBlock + threadIdx.x;
    // Every tile's range starts empty ({0, 0}); the extraction writes the
    // tiles that get pairs.
    for (uint32_t w = (uint32_t)i; w < range_words; w += gridDim.x * kBinBlock) ranges[w] = 0u;
    const bool emits = i < n && rect_count(rects[i]) > 0;
    uint32_t total;
    const uint32_t excl = block_exclusive_scan_256<uint32_t>(emits ? 1u : 0u, ws, &total);
    if (emits) {
        const size_t pos = (size_t)blk_emit_offs[blockIdx.x] + excl;
        dkeys[pos] = __float_as_uint(__ldg(depths + i));
        didx[pos] = (uint32_t)i;
    }
}

// The depth-sorted splat indices: buffer 1, or buffer 0 when a device-planned
// sort (depth_and_or set) found no varying digit and ran no pass.
__device__ __forceinline__ const uint32_t *depth_sorted(const DepthBuffers &b, const unsigned long long *depth_and_or)
{
    if (!depth_and_or) return b.v[1];
    int executed;
    field_pass(__ldg(depth_and_or) ^ __ldg(depth_and_or + 1), 0, 32, -1, &executed);
    return executed ? b.v[1] : b.v[0];
}

// Per block of 256 depth-sorted splats: their pair total.
__global__ void __launch_bounds__(kBinBlock)
k_sorted_sums(DepthBuffers dbufs, const uint2 *__restrict__ rects, int n, int m_host,
              unsigned long long *__restrict__ blk_sorted, unsigned long long *__restrict__ scalars,
              const unsigned long long *__restrict__ depth_and_or)
{
    grid_dependency_begin();
    __shared__ unsigned long long ws[8];
    // the emitting count: m_host when the host knows it, else the device's
    const int m = m_host >= 0 ? m_host : (int)min(__ldg(scalars + kScalarEmitting), (unsigned long long)n);
    const uint32_t *__restrict__ sorted_idx = depth_sorted(dbufs, depth_and_or);
    const int k = blockIdx.x * kBinBlock + threadIdx.x;
    const uint32_t c = k < m ? rect_count(rects[sorted_idx[k]]) : 0u;
    unsigned long long total;
    block_exclusive_scan_256<unsigned long long>(c, ws, &total);
    if (threadIdx.x == 0) blk_sorted[blockIdx.x] = total;
    // The last block turns the per-block sums into offsets.
    if (last_block_done(scalars + kScalarTicketSums)) block_scan_inplace_256(blk_sorted, (int)gridDim.x, ws);
}

// --- emit ------------------------------------------------------------------

// Pairs per block that the start-bit index covers; a block with more pairs
// (very large splats) finds each pair's splat by binary search instead.
constexpr int kEmitIndexPairs = 16384;

// Each block takes 256 consecutive depth-sorted splats, scans their counts and
// writes its contiguous slice of pairs with all 256 threads, so a splat with
// thousands of tiles does not serialise on one thread.  Within a splat the pairs
// go in row-major tile order; across splats in depth order.  A pair finds its
// splat as the rank of the last splat start at or before it (a bit per pair
// marks the starts; every splat here has at least one pair).  Also folds the
// AND / OR of the keys for the tile sort's plan.
__global__ void __launch_bounds__(kBinBlock)
k_emit(const uint2 *__restrict__ rects, const float *__restrict__ depths, DepthBuffers dbufs, int n, int m_host,
       int tiles_x, const unsigned long long *__restrict__ blk_offs, uint64_t *__restrict__ keys,
       uint32_t *__restrict__ vals, unsigned long long *__restrict__ scalars,
       const unsigned long long *__restrict__ depth_and_or)
{
    grid_dependency_begin();
    const int m = m_host >= 0 ? m_host : (int)min(__ldg(scalars + kScalarEmitting), (unsigned long long)n);
    const uint32_t *__restrict__ sorted_idx = depth_sorted(dbufs, depth_and_or);
    if ((int)(blockIdx.x * kBinBlock) >= m) {
        // no splat of this block emits; its part of the keys' AND / OR is empty
        return;
    }
    __shared__ uint32_t s_off[kBinBlock];
    __shared__ uint32_t s_x0y0[kBinBlock];
    __shared__ uint32_t s_w[kBinBlock];
    __shared__ float s_invw[kBinBlock];
    __shared__ uint32_t s_db[kBinBlock];
    __shared__ uint32_t s_idx[kBinBlock];
    __shared__ uint32_t s_bits[kEmitIndexPairs / 32];
    __shared__ uint32_t s_rank[kEmitIndexPairs / 32];
    __shared__ uint32_t ws[8];
    __shared__ unsigned long long s_and[8], s_or[8];

    const int k = blockIdx.x * kBinBlock + threadIdx.x;
    uint32_t c = 0, i = 0;
    uint2 pr = make_uint2(1u, 0u);
    if (k < m) {
        i = sorted_idx[k];
        pr = rects[i];
        c = rect_count(pr);
    }
    uint32_t total;
    const uint32_t excl = block_exclusive_scan_256<uint32_t>(c, ws, &total);
    const bool indexed = total <= (uint32_t)kEmitIndexPairs;
    if (indexed)
        for (uint32_t wi = threadIdx.x; wi < (total + 31) / 32; wi += kBinBlock) s_bits[wi] = 0u;
    s_off[threadIdx.x] = excl;
    s_x0y0[threadIdx.x] = pr.x;
    const uint32_t w = c ? rect_width(pr) : 1u;
    s_w[threadIdx.x] = w;
    s_invw[threadIdx.x] = 1.0f / (float)w;
    s_db[threadIdx.x] = k < m ? __float_as_uint(__ldg(depths + i)) : 0u;
    s_idx[threadIdx.x] = i;
    __syncthreads();
    if (indexed) {
        if (c) atomicOr(&s_bits[excl >> 5], 1u << (excl & 31));
        __syncthreads();
        // s_rank[w]: starts in the words before w (one warp scans the words).
        if (threadIdx.x < 32) {
            uint32_t carry = 0;
            for (uint32_t w0 = 0; w0 < (total + 31) / 32; w0 += 32) {
                const uint32_t wi = w0 + threadIdx.x;
                const uint32_t cnt = wi < (total + 31) / 32 ? __popc(s_bits[wi]) : 0u;
                uint32_t incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t t = __shfl_up_sync(kFull, incl, o);
                    if ((int)threadIdx.x >= o) incl += t;
                }
                if (wi < (total + 31) / 32) s_rank[wi] = carry + incl - cnt;
                carry += __shfl_sync(kFull, incl, 31);
            }
        }
        __syncthreads();
    }

    const unsigned long long base = blk_offs[blockIdx.x];
    unsigned long long acc_and = ~0ull, acc_or = 0ull;
    for (uint32_t q = threadIdx.x; q < total; q += kBinBlock) {
        int lo;
        if (indexed) {
            const uint32_t bits = s_bits[q >> 5] & (0xffffffffu >> (31 - (q & 31)));
            lo = (int)(s_rank[q >> 5] + __popc(bits)) - 1;
        } else {
            // Last splat t with s_off[t] <= q; it has a nonzero count.
            int l = 0, h = kBinBlock - 1;
            while (l < h) {
                const int mid = (l + h + 1) >> 1;
                if (s_off[mid] <= q) l = mid;
                else h = mid - 1;
            }
            lo = l;
        }
        const uint32_t local = q - s_off[lo];
        const uint32_t wd = s_w[lo];
        // local / wd: below 2^22 a float reciprocal is within one of the
        // quotient and one correction makes it exact.
        uint32_t dy;
        if (local < (1u << 22)) {
            dy = (uint32_t)((float)local * s_invw[lo]);
            if (dy * wd > local) --dy;
            else if ((dy + 1u) * wd <= local) ++dy;
        } else {
            dy = local / wd;
        }
        const uint32_t xy = s_x0y0[lo];
        const uint32_t ty = (xy >> 16) + dy;
        const uint32_t tx = (xy & 0xffffu) + (local - dy * wd);
        const uint64_t tile = (uint64_t)ty * (uint64_t)tiles_x + tx;
        const uint64_t key = (tile << 32) | (uint64_t)s_db[lo];
        keys[base + q] = key;
        vals[base + q] = s_idx[lo];
        acc_and &= key;
        acc_or |= key;
    }
    block_and_or_into(acc_and, acc_or, s_and, s_or, scalars + kScalarKeyAnd);
}

// --- radix sort --------------------------------------------------------------
//
// A stable LSD sort over the key bits [key_lo, key_hi), one pass per varying
// digit, each pass three kernels with no waits between CTAs:
//   upsweep  : per radix tile (256 threads x 8 or 12 keys), the count of each digit value, written
//              digit-major, counts[digit][tile], and added to totals[digit];
//   scan     : one CTA per digit value: the digit's global start (the totals of
//              all smaller digits) plus the exclusive scan of its row, written
//              to offsets[digit][tile];
//   downsweep: each tile ranks its keys stably by digit (ballot-built peer
//              masks, per-warp counters), stages them in shared memory in digit
//              order and writes every digit's keys as one contiguous run.

// Keys per thread in a radix tile of the depth sort and of the pair sort.
#ifndef GSR_RT_ITEMS_DEPTH
#define GSR_RT_ITEMS_DEPTH 8
#endif
#ifndef GSR_RT_ITEMS_PAIRS
#define GSR_RT_ITEMS_PAIRS 12
#endif
// Resident CTAs per SM the radix downsweep is compiled for (register budget).
#ifndef GSR_RT_MIN_BLOCKS
#define GSR_RT_MIN_BLOCKS 3
#endif
constexpr int kRtThreads = 256;
constexpr int kRtItemsDepth = GSR_RT_ITEMS_DEPTH;
constexpr int kRtItemsPairs = GSR_RT_ITEMS_PAIRS;

// Buffer b of the three (a select, so the kernel parameter block is not copied
// to local memory for dynamic indexing).
template <typename K>
__device__ __forceinline__ K *keys_of(const SortBuffers<K> &p, int b)
{
    return b == 0 ? p.k[0] : (b == 1 ? p.k[1] : p.k[2]);
}
template <typename K>
__device__ __forceinline__ uint32_t *vals_of(const SortBuffers<K> &p, int b)
{
    return b == 0 ? p.v[0] : (b == 1 ? p.v[1] : p.v[2]);
}

struct PassGeom {
    int shift, width, src, dst;
};

// Which digit a pass sorts on and how it learns whether the digit varies: from
// the device AND / OR of the keys (and_or set; a constant digit's pass returns
// at once), or from the plan the host made (and_or null; only passes over
// varying digits are launched).
struct PassSpec {
    const unsigned long long *and_or;
    int key_lo, key_hi, field;
    PassGeom host;
    const unsigned long long *num;  // device: the number of keys (min'd with num_max); null: num_max
    uint32_t num_max;                // the number of keys, or their bound (the buffers' capacity)
    int stride;                      // radix tiles per digit row of counts / offsets
};

// Counts and plans that earlier kernels left on the device are read through
// the read-only path (__ldg): every thread reads the same word, and the cache
// serves a warp's and the SM's requests at once, where L2-only loads would
// send every warp's request to the same L2 slice.
__device__ __forceinline__ uint32_t pass_num(const PassSpec &p)
{
    return p.num ? (uint32_t)min(__ldg(p.num), (unsigned long long)p.num_max) : p.num_max;
}

// Geometry of pass `field` of `executed` varying digits, whose position among
// them is j.
__host__ __device__ __forceinline__ PassGeom plan_geom(int key_lo, int key_hi, int field, int j, int executed)
{
    PassGeom g;
    field_geom(key_lo, key_hi, num_fields(key_lo, key_hi), field, g.shift, g.width);
    g.dst = ((executed - 1 - j) % 2 == 0) ? 1 : 2;
    g.src = (j == 0) ? 0 : (((executed - j) % 2 == 0) ? 1 : 2);
    return g;
}

// Geometry of the pass, or false when its digit is constant (skipped).
__device__ __forceinline__ bool pass_geom(const PassSpec &p, PassGeom &g)
{
    if (!p.and_or) {
        g = p.host;
        return true;
    }
    int executed;
    const int j = field_pass(__ldg(p.and_or) ^ __ldg(p.and_or + 1), p.key_lo, p.key_hi, p.field, &executed);
    if (j < 0) return false;
    g = plan_geom(p.key_lo, p.key_hi, p.field, j, executed);
    return true;
}

template <typename K, int kRtItems>
__global__ void __launch_bounds__(kRtThreads)
k_radix_upsweep(SortBuffers<K> bufs, PassSpec ps, uint32_t *__restrict__ counts, uint32_t *__restrict__ totals)
{
    grid_dependency_begin();
    PassGeom g;
    if (!pass_geom(ps, g)) return;
    const uint32_t num = pass_num(ps);
    constexpr uint32_t kRtTile = kRtThreads * kRtItems;
    const uint32_t ntiles = (num + kRtTile - 1) / kRtTile;
    const K *__restrict__ keys = keys_of(bufs, g.src);
    const uint32_t dmask = (1u << g.width) - 1u;
    __shared__ uint32_t h[256];
    uint32_t total = 0;   // this block's count of digit threadIdx.x over its tiles
    // The grid strides over the radix tiles (one tile per block when the grid
    // covers them all).
    for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        h[threadIdx.x] = 0;
        // All of the thread's keys are loaded before the first shared-memory
        // atomic, so their latencies overlap.
        const uint32_t base = tile * kRtTile;
        K kk[kRtItems];
#pragma unroll
        for (int k = 0; k < kRtItems; ++k) {
            const uint32_t i = base + k * kRtThreads + threadIdx.x;
            kk[k] = i < num ? keys[i] : (K)0;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kRtItems; ++k) {
            const uint32_t i = base + k * kRtThreads + threadIdx.x;
            if (i < num) atomicAdd(&h[(uint32_t)(kk[k] >> g.shift) & dmask], 1u);
        }
        __syncthreads();
        if (threadIdx.x <= (int)dmask) {
            const uint32_t c = h[threadIdx.x];
            counts[(size_t)threadIdx.x * ps.stride + tile] = c;
            total += c;
        }
        __syncthreads();
    }
    if (threadIdx.x <= (int)dmask && total) atomicAdd(&totals[threadIdx.x], total);
}

__global__ void __launch_bounds__(kRtThreads)
k_radix_scan(PassSpec ps, int rt_tile, const uint32_t *__restrict__ counts, const uint32_t *__restrict__ totals,
             uint32_t *__restrict__ offsets)
{
    grid_dependency_begin();
    PassGeom g;
    if (!pass_geom(ps, g)) return;
    // the radix tiles that hold keys; rows are ps.stride long
    const int ntiles = (int)((pass_num(ps) + (uint32_t)rt_tile - 1) / (uint32_t)rt_tile);
    const uint32_t digit = blockIdx.x;
    if (digit >= (1u << g.width)) return;
    __shared__ uint32_t ws[8];
    __shared__ uint32_t s_wsum[kRtThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // Global start of this digit: the totals of all smaller digits.
    uint32_t base;
    block_exclusive_scan_256<uint32_t>(threadIdx.x < digit ? totals[threadIdx.x] : 0u, ws, &base);
    const uint32_t *row = counts + (size_t)digit * ps.stride;
    uint32_t *orow = offsets + (size_t)digit * ps.stride;
    // Warp w scans the segment [seg0, seg1) of the row: first its sum (all loads
    // independent), then, after the warps' sums are exchanged, the segment in
    // runs of 32 with a carried prefix.
    const int per = ((ntiles + kRtThreads - 1) / kRtThreads) * 32;
    const int seg0 = min(ntiles, warp * per), seg1 = min(ntiles, seg0 + per);
    uint32_t part = 0;
    for (int i = seg0 + lane; i < seg1; i += 32) part += row[i];
    part = __reduce_add_sync(kFull, part);
    if (lane == 0) s_wsum[warp] = part;
    __syncthreads();
    uint32_t carry = base;
    for (int w = 0; w < warp; ++w) carry += s_wsum[w];
#pragma unroll 4
    for (int i0 = seg0; i0 < seg1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t c = i < seg1 ? row[i] : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        if (i < seg1) orow[i] = carry + incl - c;
        carry += __shfl_sync(kFull, incl, 31);
    }
}

template <typename K, int kRtItems, int kWidth>
__global__ void __launch_bounds__(kRtThreads, GSR_RT_MIN_BLOCKS)
k_radix_downsweep(SortBuffers<K> bufs, PassSpec ps, const uint32_t *__restrict__ offsets)
{
    grid_dependency_begin();
    PassGeom g;
    if (!pass_geom(ps, g)) return;
    const uint32_t num = pass_num(ps);
    const K *__restrict__ kin = keys_of(bufs, g.src);
    const uint32_t *__restrict__ vin = vals_of(bufs, g.src);
    K *__restrict__ kout = keys_of(bufs, g.dst);
    uint32_t *__restrict__ vout = vals_of(bufs, g.dst);
    const int shift = g.shift;
    constexpr uint32_t radix = 1u << kWidth, dmask = radix - 1u;

    __shared__ uint32_t wcnt[8][256];   // per-warp digit counts, then per-warp prefixes
    __shared__ uint32_t s_lstart[256];  // start of each digit's run in the staged tile
    __shared__ uint32_t s_goff[256];    // global start of each digit's run
    __shared__ uint32_t ws[8];
    constexpr int kRtTile = kRtThreads * kRtItems;
    __shared__ K s_keys[kRtTile];
    __shared__ uint32_t s_vals[kRtTile];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t ntiles = (num + kRtTile - 1) / kRtTile;
    // The grid strides over the radix tiles (one tile per block when the grid
    // covers them all).
    for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const uint32_t tbase = tile * kRtTile;
    const uint32_t tcount = min((uint32_t)kRtTile, num - tbase);

    // Warp w owns keys [w*256, w*256+256) of the tile.  They are all loaded
    // first (their latencies overlap), then ranked in 8 rounds of 32: equal
    // digits are ranked by lane within a round and by per-warp counters,
    // updated by each digit's lowest lane, across rounds.
    const uint32_t wbase = warp * (32 * kRtItems);
    K key[kRtItems];
    uint32_t val[kRtItems], rank[kRtItems];
#pragma unroll
    for (int k = 0; k < kRtItems; ++k) {
        const uint32_t i = wbase + k * 32 + lane;
        key[k] = i < tcount ? kin[tbase + i] : (K)0;
        val[k] = i < tcount ? vin[tbase + i] : 0u;
    }
    if (tid < (int)radix) {
#pragma unroll
        for (int w = 0; w < 8; ++w) wcnt[w][tid] = 0;
        s_goff[tid] = offsets[(size_t)tid * ps.stride + tile];
    }
    GSR_CANARY(11);
    __syncthreads();
    const uint32_t lanemask_lt = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < kRtItems; ++k) {
        const bool valid = wbase + k * 32 + lane < tcount;
        const uint32_t digit = (uint32_t)(key[k] >> shift) & dmask;
        const uint32_t peers = digit_peers<kWidth>(__ballot_sync(kFull, valid), digit);
        const uint32_t before = __popc(peers & lanemask_lt);
        uint32_t prior = 0;
        if (valid && before == 0) {
            prior = wcnt[warp][digit];
            wcnt[warp][digit] = prior + __popc(peers);
        }
        prior = __shfl_sync(kFull, prior, valid ? __ffs(peers) - 1 : lane);
        __syncwarp();
        rank[k] = prior + before;
    }
    GSR_CANARY(12);
    __syncthreads();
    uint32_t tot = 0;
    if (tid < (int)radix) {
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t t = wcnt[w][tid];
            wcnt[w][tid] = tot;
            tot += t;
        }
    }
    uint32_t all;
    s_lstart[tid] = block_exclusive_scan_256<uint32_t>(tot, ws, &all);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kRtItems; ++k) {
        const uint32_t i = wbase + k * 32 + lane;
        if (i < tcount) {
            const uint32_t digit = (uint32_t)(key[k] >> shift) & dmask;
            const uint32_t lpos = s_lstart[digit] + wcnt[warp][digit] + rank[k];
            s_keys[lpos] = key[k];
            s_vals[lpos] = val[k];
        }
    }
    __syncthreads();
#pragma unroll 4
    for (uint32_t i = tid; i < tcount; i += kRtThreads) {
        const K kk = s_keys[i];
        const uint32_t digit = (uint32_t)(kk >> shift) & dmask;
        const uint32_t gpos = s_goff[digit] + (i - s_lstart[digit]);
        kout[gpos] = kk;
        vout[gpos] = s_vals[i];
    }
    __syncthreads();   // the staged tile is read before the next one is staged
    }
}

// --- ranges --------------------------------------------------------------------

// Tile starts and ends where the tile field of the sorted keys changes; each
// thread compares four consecutive keys (two 16-byte loads) and their
// neighbours.
__global__ void __launch_bounds__(256)
k_extract_ranges(PairBuffers bufs, const unsigned long long *__restrict__ num_dev, uint32_t num_max,
                 uint32_t *__restrict__ ranges, const unsigned long long *__restrict__ and_or, int key_lo, int key_hi)
{
    grid_dependency_begin();
    const uint32_t num = num_dev ? (uint32_t)min(__ldg(num_dev), (unsigned long long)num_max) : num_max;
    // A tile sort that ran no pass (every key shares its tile bits) left the
    // emitted order, already sorted, in buffer 0: copy it to the result.
    const uint64_t *__restrict__ keys = bufs.k[1];
    bool copy = false;
    if (and_or) {
        int executed;
        field_pass(and_or[0] ^ and_or[1], key_lo, key_hi, -1, &executed);
        copy = executed == 0;
        if (copy) keys = bufs.k[0];
    }
    const uint32_t step = gridDim.x * blockDim.x * 4u;
    for (uint32_t i0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4u; i0 < num; i0 += step) {
        if (copy)
            for (uint32_t i = i0; i < min(i0 + 4u, num); ++i) {
                bufs.k[1][i] = bufs.k[0][i];
                bufs.v[1][i] = bufs.v[0][i];
            }
        uint32_t t[6];  // tiles of keys i0 - 1 .. i0 + 4 (0xffffffff outside [0, num))
        t[0] = i0 > 0 ? (uint32_t)(__ldg(keys + i0 - 1) >> 32) : 0xffffffffu;
        if (i0 + 4 <= num) {
            const ulonglong2 a = __ldg(reinterpret_cast<const ulonglong2 *>(keys + i0));
            const ulonglong2 b = __ldg(reinterpret_cast<const ulonglong2 *>(keys + i0 + 2));
            t[1] = (uint32_t)(a.x >> 32);
            t[2] = (uint32_t)(a.y >> 32);
            t[3] = (uint32_t)(b.x >> 32);
            t[4] = (uint32_t)(b.y >> 32);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                t[1 + k] = i0 + k < num ? (uint32_t)(__ldg(keys + i0 + k) >> 32) : 0xffffffffu;
        }
        t[5] = i0 + 4 < num ? (uint32_t)(__ldg(keys + i0 + 4) >> 32) : 0xffffffffu;
#pragma unroll
        for (int k = 1; k <= 4; ++k) {
            const uint32_t i = i0 + k - 1;
            if (i >= num) break;
            if (t[k - 1] != t[k]) ranges[2 * (size_t)t[k]] = i;
            if (t[k + 1] != t[k]) ranges[2 * (size_t)t[k] + 1] = i + 1;
        }
    }
}

// --- launch order of the tiles -----------------------------------------------

// 0 for no work, else 1 + floor(8 log2 c): 256 classes a factor 2^(1/8) apart
// (the approximate log2 only moves a tile between neighbouring classes).
__device__ __forceinline__ int cost_class(uint32_t c)
{
    return c == 0 ? 0 : min(255, 1 + (int)(8.0f * __log2f((float)c)));
}

// One block: a counting sort of the tiles by cost class, largest first.
__global__ void __launch_bounds__(1024)
k_tile_order(const uint2 *__restrict__ ranges, const uint32_t *__restrict__ costs, int num_tiles,
             uint32_t *__restrict__ order)
{
    grid_dependency_begin();
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_cursor[256];
    if (threadIdx.x < 256) s_hist[threadIdx.x] = 0;
    __syncthreads();
    auto cost_of = [&](int t) { return ranges ? ranges[t].y - ranges[t].x : costs[t]; };
    for (int t = threadIdx.x; t < num_tiles; t += blockDim.x) atomicAdd(&s_hist[cost_class(cost_of(t))], 1u);
    __syncthreads();
    if (threadIdx.x < 32) {
        // Exclusive scan over the classes from the largest down: lane l owns
        // classes 255 - 8l down to 248 - 8l.
        const int lane = threadIdx.x;
        uint32_t local[8], sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            local[k] = s_hist[255 - (8 * lane + k)];
            sum += local[k];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t run = incl - sum;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            s_cursor[255 - (8 * lane + k)] = run;
            run += local[k];
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < num_tiles; t += blockDim.x)
        order[atomicAdd(&s_cursor[cost_class(cost_of(t))], 1u)] = (uint32_t)t;
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

// Growing the arena frees buffers that queued work (of this or an earlier call)
// may still use: wait for the device first.  Growth is rare (grow-only arena).
int drain_before_free(gsr_ctx *ctx) { return cuda_check(ctx, cudaDeviceSynchronize(), "cudaDeviceSynchronize"); }

template <typename T>
int grow(gsr_ctx *ctx, T **ptr, size_t *cap, size_t need, size_t elems_per, const char *what)
{
    if (need <= *cap && *ptr) return GSR_OK;
    if (*ptr) {
        int rc = drain_before_free(ctx);
        if (rc) return rc;
        cudaFree(*ptr);
        *ptr = nullptr;
    }
    *cap = 0;
    cudaError_t e = device_alloc(ctx, (void **)ptr, std::max<size_t>(need, 1) * elems_per * sizeof(T));
    if (e != cudaSuccess) {
        cudaGetLastError();
        *ptr = nullptr;
        return fail(ctx, GSR_ERR_OOM, std::string("cudaMalloc failed for ") + what);
    }
    *cap = need;
    return GSR_OK;
}

template <typename K>
int grow_sort_buffers(gsr_ctx *ctx, SortBuffers<K> &b, size_t *cap, size_t need, const char *what)
{
    if (need <= *cap && b.k[0]) return GSR_OK;
    if (b.k[0]) {
        int rc = drain_before_free(ctx);
        if (rc) return rc;
    }
    for (int j = 0; j < 3; ++j) {
        if (b.k[j]) cudaFree(b.k[j]);
        if (b.v[j]) cudaFree(b.v[j]);
        b.k[j] = nullptr;
        b.v[j] = nullptr;
    }
    *cap = 0;
    need = std::max<size_t>(need, 1);
    for (int j = 0; j < 3; ++j) {
        if (device_alloc(ctx, (void **)&b.k[j], need * sizeof(K)) != cudaSuccess ||
            device_alloc(ctx, (void **)&b.v[j], need * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, GSR_ERR_OOM, std::string("cudaMalloc failed for ") + what);
        }
    }
    *cap = need;
    return GSR_OK;
}

#define GSR_LAUNCH(ctx, ...)                                                          \
    do {                                                                              \
        int _rc = cuda_check((ctx), launch_kernel((ctx), __VA_ARGS__), "kernel launch"); \
        if (_rc) return _rc;                                                          \
    } while (0)

// The downsweep compiled for digit width `width` (1..8 bits).
template <typename K, int kRtItems>
int launch_downsweep(gsr_ctx *ctx, int width, int ntiles, cudaStream_t stream, SortBuffers<K> bufs, PassSpec ps,
                     const uint32_t *offsets)
{
    auto go = [&](auto kernel) {
        return cuda_check(ctx, launch_kernel(ctx, kernel, dim3(ntiles), dim3(kRtThreads), stream, bufs, ps, offsets),
                          "kernel launch");
    };
    switch (width) {
    case 1: return go(k_radix_downsweep<K, kRtItems, 1>);
    case 2: return go(k_radix_downsweep<K, kRtItems, 2>);
    case 3: return go(k_radix_downsweep<K, kRtItems, 3>);
    case 4: return go(k_radix_downsweep<K, kRtItems, 4>);
    case 5: return go(k_radix_downsweep<K, kRtItems, 5>);
    case 6: return go(k_radix_downsweep<K, kRtItems, 6>);
    case 7: return go(k_radix_downsweep<K, kRtItems, 7>);
    default: return go(k_radix_downsweep<K, kRtItems, 8>);
    }
}

// Stable LSD sort of bufs buffer 0 into buffer 1 over the key bits
// [key_lo, key_hi).  num_dev: the number of keys on the device, num_max its
// bound (the buffers' capacity): the grids then hold as many blocks as the
// SMs keep resident and stride over the radix tiles; null: num_max is the
// count, and every radix tile gets its block.  and_or: the device
// AND / OR of the keys.  host_and_or: the same two values already on the host,
// or null; with them only the passes over varying digits are launched.
template <typename K, int kRtItems>
int radix_sort(gsr_ctx *ctx, SortBuffers<K> bufs, const unsigned long long *num_dev, uint32_t num_max, int key_lo,
               int key_hi, const unsigned long long *and_or, const unsigned long long *host_and_or,
               uint32_t *totals, cudaStream_t stream)
{
    int rc;
    constexpr int kRtTile = kRtThreads * kRtItems;
    const int ntiles = (int)((num_max + kRtTile - 1) / kRtTile);
    if (ntiles == 0) return GSR_OK;
    // [256][ntiles] counts, then [256][ntiles] offsets (sized by bin_splats).
    uint32_t *counts = ctx->radix_counts;
    uint32_t *offsets = ctx->radix_counts + (size_t)256 * ntiles;
    const int nf = num_fields(key_lo, key_hi);
    int executed = nf;
    if (host_and_or) {
        field_pass(host_and_or[0] ^ host_and_or[1], key_lo, key_hi, -1, &executed);
        if (executed == 0) {
            // No digit varies: the input order is the sorted order (num_max
            // keys exactly when the host planned the sort).
            if ((rc = cuda_check(ctx, cudaMemcpyAsync(bufs.k[1], bufs.k[0], (size_t)num_max * sizeof(K),
                                                      cudaMemcpyDeviceToDevice, stream), "cudaMemcpyAsync")) ||
                (rc = cuda_check(ctx, cudaMemcpyAsync(bufs.v[1], bufs.v[0], (size_t)num_max * sizeof(uint32_t),
                                                      cudaMemcpyDeviceToDevice, stream), "cudaMemcpyAsync")))
                return rc;
            return GSR_OK;
        }
    }
    const int grid = num_dev ? std::min(ntiles, ctx->num_sms * GSR_RT_MIN_BLOCKS) : ntiles;
    for (int f = 0; f < nf; ++f) {
        PassSpec ps = {and_or, key_lo, key_hi, f, {}, num_dev, num_max, ntiles};
        if (host_and_or) {
            const int j = field_pass(host_and_or[0] ^ host_and_or[1], key_lo, key_hi, f, &executed);
            if (j < 0) continue;
            ps.and_or = nullptr;
            ps.host = plan_geom(key_lo, key_hi, f, j, executed);
        }
        int sh, w;
        field_geom(key_lo, key_hi, nf, f, sh, w);
        uint32_t *tot = totals + 256 * f;
        GSR_LAUNCH(ctx, k_radix_upsweep<K, kRtItems>, dim3(grid), dim3(kRtThreads), stream, bufs, ps, counts, tot);
        GSR_LAUNCH(ctx, k_radix_scan, dim3(1 << w), dim3(kRtThreads), stream, ps, kRtTile, counts, tot, offsets);
        if ((rc = launch_downsweep<K, kRtItems>(ctx, w, grid, stream, bufs, ps, offsets))) return rc;
    }
    // A device-planned sort that runs no pass leaves the sorted order in buffer
    // 0; the caller completes it (the range extraction copies it to buffer 1).
    return GSR_OK;
}

}  // namespace

int bin_splats(gsr_ctx *ctx, const float *splats, const float *depths, int32_t n, int32_t width,
               int32_t height, cudaStream_t stream, gsr_bins *out)
{
    int rc;
    const int tiles_x = (width + kTile - 1) / kTile;
    const int tiles_y = (height + kTile - 1) / kTile;
    const size_t num_tiles = (size_t)tiles_x * tiles_y;
    const int key_hi = 32 + bits_for(num_tiles - 1);  // keys occupy bits [0, key_hi)
    // With a reservation (gsr_reserve_pairs) the call reads nothing back: the
    // arena holds the reserved pairs, the count is checked on the device, and
    // every kernel takes its key counts from the device.
    const bool sync_free = ctx->reserved_pairs > 0;

    // Fixed-size scratch, allocated once (each piece again if an earlier
    // allocation of it failed).
    auto alloc_failed = [&](cudaError_t e, const char *what) -> int {
        if (e == cudaSuccess) return GSR_OK;
        cudaGetLastError();
        return fail(ctx, GSR_ERR_OOM, std::string("cudaMalloc failed for ") + what);
    };
    if (!ctx->scalars) {
        if ((rc = alloc_failed(device_alloc(ctx, (void **)&ctx->scalars, kScalarCount * sizeof(unsigned long long)),
                               "binning scalars")))
            return rc;
        // k_count's ticket starts at zero; k_count resets it after each use
        if ((rc = cuda_check(ctx, cudaMemset(ctx->scalars, 0, kScalarCount * sizeof(unsigned long long)),
                             "cudaMemset"))) {
            cudaFree(ctx->scalars);
            ctx->scalars = nullptr;
            return rc;
        }
    }
    if (!ctx->host_total &&
        (rc = alloc_failed(cudaHostAlloc(&ctx->host_total, 4 * sizeof(unsigned long long), cudaHostAllocDefault),
                           "pinned pair count")))
        return rc;
    if (!ctx->radix_totals &&
        (rc = alloc_failed(device_alloc(ctx, (void **)&ctx->radix_totals, 2 * 4 * 256 * sizeof(uint32_t)),
                           "radix digit totals")))
        return rc;
    const int nblk = (n + kBinBlock - 1) / kBinBlock;
    if (!ctx->depth.k[0] || (size_t)n > ctx->cap_splats) {
        size_t cap = 0;
        if ((rc = grow_sort_buffers(ctx, ctx->depth, &cap, (size_t)n, "depth sort buffers"))) return rc;
        ctx->cap_splats = 0;  // regrow the rectangles below to the same capacity
        if ((rc = grow(ctx, &ctx->rects, &ctx->cap_splats, cap, 1, "tile rectangles"))) return rc;
    }
    // Five per-block arrays: [0, c) pair sums, [c, 2c) emitting counts then
    // offsets, [2c, 3c) pair sums in depth order then offsets, [3c, 5c) the
    // AND / OR of the emitting splats' depth bits.
    if ((rc = grow(ctx, &ctx->blk_sums, &ctx->cap_blocks, (size_t)std::max(nblk, 1), 5, "block sums"))) return rc;
    unsigned long long *blk_pairs = ctx->blk_sums;
    unsigned long long *blk_emit = ctx->blk_sums + ctx->cap_blocks;
    unsigned long long *blk_sorted = ctx->blk_sums + 2 * ctx->cap_blocks;
    unsigned long long *blk_and = ctx->blk_sums + 3 * ctx->cap_blocks;
    unsigned long long *blk_or = ctx->blk_sums + 4 * ctx->cap_blocks;
    // Per tile: {start, end}, then the launch order after all tiles' ranges.
    if ((rc = grow(ctx, &ctx->ranges, &ctx->cap_tiles, num_tiles, 3, "tile ranges"))) return rc;
    ctx->tile_order = ctx->ranges + 2 * ctx->cap_tiles;

    // The pair buffers: max(65536, 16 n, 1.5 x pairs) ("C0 resident arena": grow,
    // never shrink).  Without a reservation the count is read first.
    auto grow_pairs = [&](uint64_t need, bool headroom) -> int {
        if (need <= ctx->cap_pairs && ctx->pairs.k[0]) return GSR_OK;
        size_t cap = std::max<size_t>(65536, (size_t)16 * (size_t)n);
        cap = std::max<size_t>(cap, (size_t)need + (headroom ? need / 2 : 0));
        cap = std::min<size_t>(cap, (size_t)GSR_MAX_PAIRS);
        cap = std::max<size_t>(cap, (size_t)need);
        size_t have = 0;
        if (int r = grow_sort_buffers(ctx, ctx->pairs, &have, cap, "tile pairs")) {
            ctx->cap_pairs = 0;
            return r;
        }
        ctx->cap_pairs = cap;
        return GSR_OK;
    };
    if (sync_free && (rc = grow_pairs(ctx->reserved_pairs, false))) return rc;

    // 1. counts, totals; without a reservation, read the pair total, the
    //    emitting count and the depth bits' AND / OR (the one host sync).
    uint64_t total = 0, emitting = 0;
    // (with no splats, one block still writes the zero counts)
    GSR_LAUNCH(ctx, k_count, dim3(std::max(nblk, 1)), dim3(kBinBlock), stream, splats, depths, n, tiles_x, tiles_y,
               ctx->rects, blk_pairs, blk_emit, blk_and, blk_or, ctx->scalars, ctx->radix_totals, 2 * 4 * 256,
               sync_free ? (unsigned long long)ctx->cap_pairs : (unsigned long long)GSR_MAX_PAIRS);
    if (n > 0) {
        if (!sync_free) {
            // Pair total, emitting count and the AND / OR of the emitting
            // splats' depth bits (scalar slots 0..3).
            if ((rc = cuda_check(ctx, cudaMemcpyAsync(ctx->host_total, ctx->scalars, 4 * sizeof(unsigned long long),
                                                      cudaMemcpyDeviceToHost, stream),
                                 "cudaMemcpyAsync")))
                return rc;
            if ((rc = cuda_check(ctx, cudaStreamSynchronize(stream), "cudaStreamSynchronize"))) return rc;
            total = ctx->host_total[0];
            emitting = ctx->host_total[1];
        }
    }
    if (!sync_free) {
        if (total > (uint64_t)GSR_MAX_PAIRS)
            return fail(ctx, GSR_ERR_TOO_MANY_PAIRS,
                        "tile-pair count " + std::to_string(total) + " exceeds GSR_MAX_PAIRS");
        if ((rc = grow_pairs(total, true))) return rc;
    }
    // Bounds of the key counts (exact when they were read back).
    const uint32_t num_max = sync_free ? (uint32_t)ctx->cap_pairs : (uint32_t)total;
    const uint32_t m_max = sync_free ? (uint32_t)n : (uint32_t)emitting;

    // Radix counts and offsets for the larger of the two sorts, allocated before
    // any kernel that uses them is queued.
    {
        constexpr size_t td = kRtThreads * kRtItemsDepth, tp = kRtThreads * kRtItemsPairs;
        const size_t rtiles = std::max<size_t>((m_max + td - 1) / td, (num_max + tp - 1) / tp);
        if ((rc = grow(ctx, &ctx->radix_counts, &ctx->cap_radix_tiles, std::max<size_t>(rtiles, 1), 512,
                       "radix counts")))
            return rc;
    }

    if (num_max == 0 || m_max == 0) {
        // nothing to sort: every tile's range is empty
        if ((rc = cuda_check(ctx, cudaMemsetAsync(ctx->ranges, 0, num_tiles * 2 * sizeof(uint32_t), stream),
                             "cudaMemsetAsync")))
            return rc;
    } else {
        // 3. depth sort of the emitting splats (k_compact also empties every
        //    tile's range).
        GSR_LAUNCH(ctx, k_compact, dim3(nblk), dim3(kBinBlock), stream, ctx->rects, depths, n, blk_emit,
                   ctx->depth.k[0], ctx->depth.v[0], ctx->ranges, (uint32_t)(num_tiles * 2));
        if ((rc = radix_sort<uint32_t, kRtItemsDepth>(ctx, ctx->depth,
                                                      sync_free ? ctx->scalars + kScalarEmitting : nullptr, m_max, 0, 32,
                                                      ctx->scalars + kScalarDepthAnd,
                                                      sync_free ? nullptr : ctx->host_total + 2, ctx->radix_totals,
                                                      stream)))
            return rc;
        // 4. pair offsets in depth order, emission.
        const int mblk = (int)((m_max + kBinBlock - 1) / kBinBlock);
        const unsigned long long *depth_plan = sync_free ? ctx->scalars + kScalarDepthAnd : nullptr;
        const int m_host = sync_free ? -1 : (int)m_max;
        GSR_LAUNCH(ctx, k_sorted_sums, dim3(mblk), dim3(kBinBlock), stream, ctx->depth, ctx->rects, n, m_host,
                   blk_sorted, ctx->scalars, depth_plan);
        GSR_LAUNCH(ctx, k_emit, dim3(mblk), dim3(kBinBlock), stream, ctx->rects, depths, ctx->depth, n, m_host,
                   tiles_x, blk_sorted, ctx->pairs.k[0], ctx->pairs.v[0], ctx->scalars, depth_plan);
        // 5. stable sort on the tile digits only (a sort that runs no pass,
        //    one tile included, is completed by the range extraction).
        const unsigned long long *num_dev = sync_free ? ctx->scalars + kScalarNum : nullptr;
        if ((rc = radix_sort<uint64_t, kRtItemsPairs>(ctx, ctx->pairs, num_dev, num_max, 32,
                                                      key_hi, ctx->scalars + kScalarKeyAnd, nullptr,
                                                      ctx->radix_totals + 4 * 256, stream)))
            return rc;
        // 6. per-tile ranges.
        const int xgrid = (int)((num_max + 1023) / 1024);
        GSR_LAUNCH(ctx, k_extract_ranges, dim3(sync_free ? std::min(xgrid, ctx->num_sms * 8) : xgrid), dim3(256),
                   stream, ctx->pairs, num_dev, num_max, ctx->ranges,
                   (const unsigned long long *)(ctx->scalars + kScalarKeyAnd), 32, key_hi);
    }

    // 7. the forward's launch order: longest tile lists first.
    if ((rc = launch_tile_order(ctx, ctx->ranges, nullptr, (int)num_tiles, ctx->tile_order, stream))) return rc;

    ctx->last_stream = stream;
    ctx->last_sync_free = sync_free;
    ++ctx->bin_calls;
    ctx->last_key_hi = key_hi;
    out->keys = ctx->pairs.k[1];
    out->sorted_idx = ctx->pairs.v[1];
    out->tile_ranges = ctx->ranges;
    out->tile_order = ctx->tile_order;
    out->num_pairs_dev = reinterpret_cast<const uint32_t *>(ctx->scalars + kScalarResult);
    out->num_pairs = sync_free ? GSR_PAIRS_ON_DEVICE : (uint32_t)total;
    out->n = n;
    out->width = width;
    out->height = height;
    out->tiles_x = tiles_x;
    out->tiles_y = tiles_y;
    return GSR_OK;
}

// The last binning's pair count and status from the device (waits for its
// stream).
int bin_result(gsr_ctx *ctx, uint32_t *count, uint32_t *status, uint32_t *emitting)
{
    *count = 0;
    *status = GSR_OK;
    if (emitting) *emitting = 0;
    if (!ctx->scalars) return GSR_OK;
    int rc = cuda_check(ctx, cudaStreamSynchronize(ctx->last_stream), "cudaStreamSynchronize");
    if (rc) return rc;
    unsigned long long sc[kScalarCount];
    if ((rc = cuda_check(ctx, cudaMemcpy(sc, ctx->scalars, sizeof sc, cudaMemcpyDeviceToHost), "cudaMemcpy")))
        return rc;
    const uint32_t *res = reinterpret_cast<const uint32_t *>(sc + kScalarResult);
    *count = res[0];
    *status = res[1];
    if (emitting) *emitting = (uint32_t)sc[kScalarEmitting];
    return GSR_OK;
}

// Which radix digits the last binning sorted (host side of the same rule the
// kernels apply to the AND / OR of the keys).
int bin_pass_masks(gsr_ctx *ctx, uint32_t *depth_mask, uint32_t *tile_mask, int *tile_digit_bits,
                   int *tile_digits)
{
    *depth_mask = *tile_mask = 0;
    *tile_digits = num_fields(32, ctx->last_key_hi);
    *tile_digit_bits = *tile_digits ? (ctx->last_key_hi - 32 + *tile_digits - 1) / *tile_digits : 0;
    if (!ctx->scalars) return GSR_OK;
    unsigned long long sc[kScalarCount];
    int rc = cuda_check(ctx, cudaMemcpy(sc, ctx->scalars, sizeof sc, cudaMemcpyDeviceToHost), "cudaMemcpy");
    if (rc) return rc;
    if (sc[kScalarNum] == 0) return GSR_OK;   // nothing was sorted
    for (int f = 0; f < 4; ++f) {
        int sh, w;
        field_geom(0, 32, 4, f, sh, w);
        if (field_varies(sc[kScalarDepthAnd] ^ sc[kScalarDepthOr], sh, w)) *depth_mask |= 1u << f;
    }
    for (int f = 0; f < *tile_digits; ++f) {
        int sh, w;
        field_geom(32, ctx->last_key_hi, *tile_digits, f, sh, w);
        if (field_varies(sc[kScalarKeyAnd] ^ sc[kScalarKeyOr], sh, w)) *tile_mask |= 1u << f;
    }
    return GSR_OK;
}

int launch_tile_order(gsr_ctx *ctx, const uint32_t *ranges, const uint32_t *costs, int num_tiles, uint32_t *order,
                      cudaStream_t stream)
{
    if (num_tiles <= 0) return GSR_OK;
    return cuda_check(ctx, launch_kernel(ctx, k_tile_order, dim3(1), dim3(1024), stream,
                                         reinterpret_cast<const uint2 *>(ranges), costs, num_tiles, order),
                      "tile order launch");
}

}  // namespace gsr
