// The context behind the C ABI's opaque gsr_ctx: options, the grow-only
// arena and the state the calls share.  Host code only; no kernel reads it.
#pragma once

struct gsr_ctx {
    int device = 0;
    std::string err;
    uint64_t launches = 0;
    int opt_warp_skip = 1;
    int opt_last_contrib = 1;
    int opt_warp_cull = 1;
    int opt_pdl = 1;
    int opt_deterministic = 0;
    int opt_bwd_per_splat = 0;
    int opt_split = 1;
    int opt_split_forward = 0;
    int fail_next_alloc = 0;                    // test hook: the next device allocation fails
    int num_sms = 0;                            // multiprocessors of the device (read by gsr_create)

    // Grow-only arena.
    size_t cap_pairs = 0;
    gsr::PairBuffers pairs = {};
    size_t cap_splats = 0;
    uint2 *rects = nullptr;                     // [cap_splats] packed tile rectangle per splat
    gsr::DepthBuffers depth = {};               // [cap_splats] x 3: depth sort of emitting splats
    size_t cap_blocks = 0;
    unsigned long long *blk_sums = nullptr;     // [3 * cap_blocks]: see bin.cu
    size_t cap_tiles = 0;
    uint32_t *ranges = nullptr;                 // [2 * cap_tiles]
    uint32_t *tile_order = nullptr;             // [cap_tiles] forward launch order (pair count)
    size_t cap_bwd_tiles = 0;
    uint32_t *bwd_tile_cost = nullptr;          // [cap_bwd_tiles] largest last_contributor per tile
    uint32_t *bwd_tile_order = nullptr;         // [cap_bwd_tiles] backward launch order
    size_t cap_radix_tiles = 0;
    uint32_t *radix_counts = nullptr;           // [512 * cap_radix_tiles] digit counts and offsets
    uint32_t *radix_totals = nullptr;           // [2 * 4 * 256] digit totals of both sorts
    unsigned long long *scalars = nullptr;      // see bin.cu (kScalar*)
    unsigned long long *host_total = nullptr;   // pinned: pairs, emitting, depth-bit AND / OR
    size_t cap_grad_acc = 0;
    double *grad_acc = nullptr;                 // [9 * cap] backward accumulator
    bool grad_acc_zero = false;                 // grad_acc holds zeros when no call is in flight
    size_t cap_det = 0;
    uint2 *det_escale = nullptr;                // [cap_det] fixed-point exponents (deterministic backward)
    uint32_t *det_maxima = nullptr;             // after det_escale: per-block maxima of the bounds (raster.cu)

    // Pairs reserved by gsr_reserve_pairs (0: none; the binning reads its
    // count back and sizes the arena to it).
    uint64_t reserved_pairs = 0;

    // Split backward (raster.cu): the forward records every pixel's state at
    // each segment boundary of long lists; the backward runs each segment of a
    // long list as its own CTA from that state.
    size_t cap_bnd = 0;
    float4 *bnd = nullptr;                      // [cap_bnd * 256] boundary states (S, T)
    float4 *bnd_chunk = nullptr;                // after bnd: [cap_bnd * 256] the forward split's chunk states
    uint32_t *bnd_last = nullptr;               // then [cap_bnd * 256] their last composites
    // Forward split (raster.cu): chunks past the head of crowded lists.
    size_t cap_fwd_items = 0;
    uint2 *fwd_items = nullptr;                 // [cap_fwd_items] (tile, chunk)
    size_t cap_fwd_tickets = 0;
    uint32_t *fwd_queue = nullptr;              // after fwd_items: item count, replay ticket, then a
                                                // ticket per tile ([cap_fwd_tickets]); zero between calls
    bool fwd_queue_dirty = false;               // a forward failed between queueing and clearing
    size_t cap_items = 0;
    uint2 *bwd_items = nullptr;                 // [cap_items] (tile, segment) work items in launch order
    // The forward whose boundary states bnd holds (the backward splits only
    // over the same bins and the same forward outputs).
    bool fwd_bnd_valid = false;
    uint64_t fwd_bin_call = 0;
    const float *fwd_final_T = nullptr;
    const uint32_t *fwd_last = nullptr;
    uint64_t fwd_pairs_bound = 0;
    uint64_t bin_calls = 0;                     // gsr_bin_splats calls made

    // Last binning, for gsr_get_bin_stats and gsr_num_pairs.
    cudaStream_t last_stream = nullptr;
    bool last_sync_free = false;                // its counts stayed on the device
    int last_key_hi = 32;                       // keys occupied bits [0, last_key_hi)
};
