"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare them."""
import numpy as np
import torch

import oracle

# Relative uncertainty of one exponential between the two sides: the kernel's
# expf is within 2 ulp, the oracle's correctly rounded, so 2.5 ulp apart at
# most; doubled.  The kernel evaluates sigma in the oracle's operation order
# with one rounding per operation, so sigma itself carries no uncertainty.
EPS_ALPHA = 6e-7
SIGMA_ULPS = 0.0
FWD_TOL = 1e-5          # absolute, per channel of out_rgbw and final_T
GRAD_ATOL = 1e-4        # |g - g_ref| <= GRAD_ATOL + GRAD_RTOL |g_ref| + GRAD_COND sum|t|
GRAD_RTOL = 1e-4
# A gradient is a sum of per-pixel terms t.  A float evaluation of each term
# carries a few roundings, so its error is bounded by about k u sum|t|
# (u = 2^-24).  When the terms cancel (sum|t| >> |sum t|, condition numbers of
# 1e4 and more occur for the conic of large elongated splats) that bound, not
# 1e-4, is what any float implementation can promise; k = 8.
GRAD_COND = 8 * 2.0 ** -24


def to_dev(a, dev="cuda:0"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_gpu(gsr, ctx, wl, backward=True, dev="cuda:0"):
    sp, dp, dl = to_dev(wl.splats, dev), to_dev(wl.depths, dev), to_dev(wl.dl_dout, dev)
    bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
    res = {"keys": bins.keys().cpu().numpy().view(np.uint64),
           "idx": bins.sorted_idx().cpu().numpy().view(np.uint32),
           "ranges": bins.tile_ranges().cpu().numpy().view(np.uint32),
           "num_pairs": bins.num_pairs}
    out, final_t, last = gsr.rasterize_forward(ctx, sp, bins)
    res["out"] = out.cpu().numpy()
    res["final_T"] = final_t.cpu().numpy()
    res["last"] = last.cpu().numpy().view(np.uint32)
    if backward:
        grad = gsr.rasterize_backward(ctx, sp, bins, dl, final_t, last)
        res["grad"] = grad.cpu().numpy()
    torch.cuda.synchronize()
    return res


def run_oracle(wl, backward=True):
    keys, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    f = oracle.forward(wl.splats, idx, ranges, wl.width, wl.height, eps_alpha=EPS_ALPHA,
                       sigma_ulps=SIGMA_ULPS)
    res = {"keys": keys, "idx": idx, "ranges": ranges, "fwd": f}
    if backward:
        res["bwd"] = oracle.backward(wl.splats, idx, ranges, wl.width, wl.height, wl.dl_dout,
                                     eps_alpha=EPS_ALPHA, sigma_ulps=SIGMA_ULPS)
    return res


def check_bins(g, o):
    assert g["num_pairs"] == len(o["keys"])
    assert np.array_equal(g["keys"], o["keys"]), "sorted keys differ"
    assert np.array_equal(g["idx"], o["idx"]), "sorted indices differ"
    assert np.array_equal(g["ranges"], o["ranges"]), "tile ranges differ"


def check_forward(g, o, max_knife_frac=2e-3):
    f = o["fwd"]
    knife = f["margin"] < 1.0
    d = np.max(np.abs(g["out"] - f["out"]), axis=1)
    d = np.maximum(d, np.abs(g["final_T"] - f["final_T"]))
    bad = (d > FWD_TOL) | (g["last"] != f["last"])
    unexplained = np.nonzero(bad & ~knife)[0]
    assert unexplained.size == 0, (
        f"{unexplained.size} pixels differ away from any threshold knife-edge; first "
        f"{unexplained[:5]}: |d| {d[unexplained[:5]]}, last gpu {g['last'][unexplained[:5]]} "
        f"oracle {f['last'][unexplained[:5]]}")
    assert bad.sum() <= max(4, max_knife_frac * bad.size)
    return {"max_abs": float(d[~knife].max()) if (~knife).any() else 0.0,
            "knife_px": int(knife.sum()), "knife_diff_px": int(bad.sum())}


def check_backward(g, o, max_knife_frac=5e-3):
    b = o["bwd"]
    ref = b["grad"]
    diff = np.abs(g["grad"].astype(np.float64) - ref)
    plain_tol = GRAD_ATOL + GRAD_RTOL * np.abs(ref)
    bad = np.any(diff > plain_tol + GRAD_COND * b["gabs"], axis=1)
    cond_used = int(np.sum(diff > plain_tol))
    unexplained = np.nonzero(bad & ~b["knife"])[0]
    assert unexplained.size == 0, (
        f"{unexplained.size} splats' gradients differ away from knife-edges; first "
        f"{unexplained[:5]}: gpu {g['grad'][unexplained[:1]]} oracle {ref[unexplained[:1]]}")
    assert bad.sum() <= max(4, max_knife_frac * bad.size)
    ok = ~b["knife"]
    rel = diff[ok] / (np.abs(ref[ok]) + 1e-3)
    return {"max_abs": float(diff[ok].max()) if ok.any() else 0.0,
            "max_rel": float(rel.max()) if ok.any() else 0.0,
            "knife_splats": int(b["knife"].sum()), "knife_diff_splats": int(bad.sum()),
            "components_beyond_1e-4_within_cond_bound": cond_used}


def varying_digit_mask(keys, lo, hi, ndigits):
    """Bit f set when digit f of the key bits [lo, hi), split into ndigits equal
    digits, is not the same in every key (computed from the oracle's keys)."""
    if len(keys) == 0 or ndigits == 0:
        return 0
    k = keys.astype(np.uint64)
    diff = int(np.bitwise_and.reduce(k) ^ np.bitwise_or.reduce(k))
    w = (hi - lo + ndigits - 1) // ndigits
    mask = 0
    for f in range(ndigits):
        sh = lo + f * w
        width = min(w, hi - sh)
        if (diff >> sh) & ((1 << width) - 1):
            mask |= 1 << f
    return mask
