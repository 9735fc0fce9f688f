"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare them."""
import numpy as np
import torch

import oracle

# Relative uncertainty of one exponential between the two sides: the kernels'
# split exponential is within 3 ulp of the correctly rounded value and the
# oracle's within half an ulp, so 3.5 ulp (2.1e-7) apart at most; about
# tripled.  The kernels evaluate sigma in the oracle's operation order with one
# rounding per operation, so sigma itself carries no uncertainty.
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


def as_result(out, final_t, last, grad=None):
    """The parity checks' view of one forward (and backward) run on the GPU."""
    torch.cuda.synchronize()
    res = {"out": out.cpu().numpy(), "final_T": final_t.cpu().numpy(), "last": last.cpu().numpy().view(np.uint32)}
    if grad is not None:
        res["grad"] = grad.cpu().numpy() if isinstance(grad, torch.Tensor) else np.asarray(grad)
    return res


def record_stats(name, **stats):
    """Appends the parity statistics of one case to the JSON-lines file named by
    GSR_PARITY_STATS, when that is set."""
    import json
    import os
    path = os.environ.get("GSR_PARITY_STATS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, **stats}) + "\n")


def run_oracle(wl, backward=True):
    keys, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    f = oracle.forward(wl.splats, idx, ranges, wl.width, wl.height, eps_alpha=EPS_ALPHA,
                       sigma_ulps=SIGMA_ULPS)
    res = {"keys": keys, "idx": idx, "ranges": ranges, "fwd": f, "wl": wl}
    if backward:
        res["bwd"] = oracle.backward(wl.splats, idx, ranges, wl.width, wl.height, wl.dl_dout,
                                     eps_alpha=EPS_ALPHA, sigma_ulps=SIGMA_ULPS)
    return res


def check_bins(g, o):
    assert g["num_pairs"] == len(o["keys"])
    assert np.array_equal(g["keys"], o["keys"]), "sorted keys differ"
    assert np.array_equal(g["idx"], o["idx"]), "sorted indices differ"
    assert np.array_equal(g["ranges"], o["ranges"]), "tile ranges differ"


# --- knife-edges: differences explained by forced decisions ------------------
#
# A threshold decision (alpha against 1/255, next_T against 1e-4, raw against
# 0.999) whose tested value lies within its rounding uncertainty of the
# threshold may be taken the other way by a correct float implementation.  A
# pixel or a splat that differs from the oracle beyond tolerance passes only if
# the oracle, re-run with such decisions taken the other way (a forced replay,
# which refuses any flip of a decision outside its uncertainty), reproduces the
# GPU's result within the same tolerance.  Nothing is excused by a flag alone.

def _fwd_diff(g, out, final_t):
    d = np.max(np.abs(g["out"].astype(np.float64) - out), axis=1)
    return np.maximum(d, np.abs(g["final_T"].astype(np.float64) - final_t))


def explain_pixel(wl, o, g, p, tol=FWD_TOL, max_tries=64, max_depth=3):
    """The flips (pos, type) of pixel p under which the oracle's forced replay
    gives g's colour, w and final_T within tol and g's last_contrib, or None.
    Breadth first over the decisions within their uncertainty along each
    replay, fewest flips first."""
    px, py = int(p % wl.width), int(p // wl.width)
    g_out = g["out"][p].astype(np.float64)
    g_T, g_last = float(g["final_T"][p]), int(g["last"][p])
    frontier, seen, tries = [()], {()}, 0
    while frontier:
        nxt = []
        for F in frontier:
            if tries >= max_tries:
                return None
            tries += 1
            table = oracle.flip_table([(p, pos, typ) for pos, typ in F])
            out5, last, dec, refused = oracle.pixel_forced(wl.splats, o["idx"], o["ranges"], wl.width,
                                                           wl.height, px, py, table, eps_alpha=EPS_ALPHA,
                                                           sigma_ulps=SIGMA_ULPS)
            d = max(np.max(np.abs(out5[:4].astype(np.float64) - g_out)), abs(float(out5[4]) - g_T))
            if refused == 0 and d <= tol and last == g_last:
                return F
            if len(F) >= max_depth:
                continue
            for dd in np.sort(dec, order="margin"):
                c = (int(dd["pos"]), int(dd["type"]))
                if c in F:
                    continue
                key = tuple(sorted(F + (c,)))
                if key not in seen:
                    seen.add(key)
                    nxt.append(key)
        frontier = nxt
    return None


def forward_flips(g, o, tol=FWD_TOL):
    """Flip table that explains every pixel where g's forward differs from the
    oracle's (cached in o), and the pixels no flips explain."""
    if o.get("_flips_of") is g:
        return o["fwd_flips"], o["fwd_unexplained"]
    wl, f = o["wl"], o["fwd"]
    d = _fwd_diff(g, f["out"], f["final_T"])
    bad = np.nonzero((d > tol) | (g["last"] != f["last"]))[0]
    entries, unexplained = [], []
    for p in bad:
        F = explain_pixel(wl, o, g, int(p), tol) if f["margin"][p] < 1.0 else None
        if F is None:
            unexplained.append(int(p))
        else:
            entries += [(int(p), pos, typ) for pos, typ in F]
    o["_flips_of"], o["fwd_flips"], o["fwd_unexplained"] = g, oracle.flip_table(entries), unexplained
    return o["fwd_flips"], unexplained


def check_forward(g, o, tol=FWD_TOL):
    """g's forward against the oracle: every pixel within tol (colour, w,
    final_T) with the same last_contrib, where the oracle takes the decisions
    that a forced replay shows g took."""
    wl, f = o["wl"], o["fwd"]
    flips, unexplained = forward_flips(g, o, tol)
    d0 = _fwd_diff(g, f["out"], f["final_T"])
    assert not unexplained, (
        f"{len(unexplained)} pixels differ and no decisions within rounding explain them; first "
        f"{unexplained[:5]}: |d| {d0[unexplained[:5]]}, margin {f['margin'][unexplained[:5]]}, last gpu "
        f"{g['last'][unexplained[:5]]} oracle {f['last'][unexplained[:5]]}")
    if len(flips):
        ff = oracle.forward_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, flips,
                                   eps_alpha=EPS_ALPHA, sigma_ulps=SIGMA_ULPS)
        assert ff["refused"] == 0
        d = _fwd_diff(g, ff["out"], ff["final_T"])
        assert np.all(d <= tol) and np.array_equal(g["last"], ff["last"]), "the forced replay does not hold"
    else:
        d = d0
    return {"max_abs": float(d.max()) if d.size else 0.0, "knife_px": int(np.sum(f["margin"] < 1.0)),
            "flipped_px": int(len(np.unique(flips["pixel"]))) if len(flips) else 0,
            "flips": int(len(flips))}


def _grad_tol(ref, gabs):
    return GRAD_ATOL + GRAD_RTOL * np.abs(ref) + GRAD_COND * gabs


def explain_splat(wl, o, g, flips, s, ref_s, gabs_s, max_cands=20):
    """Flips of splat s's own alpha and clamp decisions (within their
    uncertainty, and consistent with g's last_contrib at their pixel) under
    which its forced gradient matches g's; [] if none is needed, None if no
    such set is found.  A flip at one pixel changes only that pixel's terms,
    so each candidate's effect is its pixel's change, and the subsets are
    searched over those effects; the caller re-checks the chosen flips with a
    full forced replay."""
    cands, margins = oracle.splat_decisions(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, flips,
                                            s, eps_alpha=EPS_ALPHA, sigma_ulps=SIGMA_ULPS)
    keep = []
    for c, m in sorted(zip(cands, margins), key=lambda cm: cm[1]):
        p, pos, typ = int(c["pixel"]), int(c["pos"]), int(c["type"])
        if typ == oracle.DEC_ALPHA and not pos + 1 < int(g["last"][p]):
            continue        # this flip would move the pixel's last_contrib
        if typ == oracle.DEC_STOP:
            continue        # so would this one
        keep.append((p, pos, typ))
    keep = keep[:max_cands]
    target = g["grad"][s].astype(np.float64) - ref_s
    if not keep:
        return None
    deltas = []
    for p, pos, typ in keep:
        px, py = p % wl.width, p // wl.width
        a, _ = oracle.pixel_backward_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, wl.dl_dout,
                                            px, py, flips, s, eps_alpha=EPS_ALPHA, sigma_ulps=SIGMA_ULPS)
        both = oracle.flip_table(list(map(tuple, flips[flips["pixel"] == p][["pixel", "pos", "type"]].tolist()))
                                 + [(p, pos, typ)])
        b, refused = oracle.pixel_backward_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height,
                                                  wl.dl_dout, px, py, both, s, eps_alpha=EPS_ALPHA,
                                                  sigma_ulps=SIGMA_ULPS)
        deltas.append(b - a if refused == 0 else np.full(9, np.inf))
    deltas = np.array(deltas)
    k = len(keep)

    def score(mask):
        tot = deltas[mask].sum(axis=0) if mask.any() else np.zeros(9)
        return float(np.max(np.abs(target - tot) / _grad_tol(ref_s + tot, gabs_s)))

    if k <= 12:
        masks = ((np.arange(1 << k)[:, None] >> np.arange(k)) & 1).astype(bool)
        scores = [score(m) for m in masks[1:]]
        best = int(np.argmin(scores)) + 1
        chosen = masks[best]
        if scores[best - 1] > 1.0:
            return None
    else:
        chosen = np.zeros(k, dtype=bool)
        cur = score(chosen)
        while cur > 1.0:
            trial = []
            for i in np.nonzero(~chosen)[0]:
                m = chosen.copy()
                m[i] = True
                trial.append((score(m), i))
            if not trial:
                return None
            sc, i = min(trial)
            if sc >= cur:
                return None
            chosen[i] = True
            cur = sc
    return [keep[i] for i in np.nonzero(chosen)[0]]


def check_backward(g, o, cond_cap=None):
    """g's gradients against the oracle's, each splat within
    GRAD_ATOL + GRAD_RTOL |g_ref| + GRAD_COND sum|t|, where the oracle takes the
    forward decisions a forced replay shows g took (g must carry the forward's
    outputs the gradients were computed from) and, for a splat still off, the
    flips of its own alpha or clamp decisions that explain it.  cond_cap: the
    most components allowed to need the GRAD_COND term."""
    wl, b = o["wl"], o["bwd"]
    flips, unexplained = forward_flips(g, o)
    assert not unexplained, f"{len(unexplained)} pixels of the forward are not explained: {unexplained[:5]}"
    grad = g["grad"].astype(np.float64)

    def forced(table):
        if len(table) == 0:
            return b["grad"], b["gabs"]
        r = oracle.backward_forced(wl.splats, o["idx"], o["ranges"], wl.width, wl.height, wl.dl_dout, table,
                                   eps_alpha=EPS_ALPHA, sigma_ulps=SIGMA_ULPS)
        assert r["refused"] == 0
        return r["grad"], r["gabs"]

    ref, gabs = forced(flips)
    bad = np.nonzero(np.any(np.abs(grad - ref) > _grad_tol(ref, gabs), axis=1))[0]
    extra, unexplained_s = [], []
    for s in bad:
        F = explain_splat(wl, o, g, flips, int(s), ref[s], gabs[s])
        if F is None:
            unexplained_s.append(int(s))
        else:
            extra += F
    assert not unexplained_s, (
        f"{len(unexplained_s)} splats' gradients differ and no decisions within rounding explain them; "
        f"first {unexplained_s[:3]}: gpu {g['grad'][unexplained_s[:1]]} oracle {ref[unexplained_s[:1]]}")
    if extra:
        flips = oracle.flip_table(list(map(tuple, flips[["pixel", "pos", "type"]].tolist())) + extra)
        ref, gabs = forced(flips)
    diff = np.abs(grad - ref)
    plain_tol = GRAD_ATOL + GRAD_RTOL * np.abs(ref)
    over = diff > plain_tol + GRAD_COND * gabs
    assert not over.any(), (f"{int(over.any(axis=1).sum())} splats fail with every flip applied; first "
                            f"{np.nonzero(over.any(axis=1))[0][:3]}")
    cond_used = int(np.sum(diff > plain_tol))
    if cond_cap is not None:
        assert cond_used <= cond_cap, f"{cond_used} components needed the GRAD_COND term (cap {cond_cap})"
    rel = diff / (np.abs(ref) + 1e-3)
    return {"max_abs": float(diff.max()) if diff.size else 0.0, "max_rel": float(rel.max()) if rel.size else 0.0,
            "knife_splats": int(b["knife"].sum()), "flips": int(len(flips)), "hidden_flips": len(extra),
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
