"""A CPU model of the heavy-tile split, against the oracle.

Splitting one tile's list across CTAs has to keep the early stop (T < 1e-4).
A chunk cannot know the transmittance in front of it, so chunks composite
from T = 1 without stopping and record their colour C_k, their transmittance
product P_k and their last composite.  A merge then walks each pixel's chunks
in order.  While T_in P_k stays at or above 1e-4, no stop can fall inside
chunk k (the running product only decreases), so (C, T) <- (C + T_in C_k,
T_in P_k).  Otherwise the pixel stops inside chunk k, which is replayed.

Two models: the design study (`_split_forward`: segments of any length from
the list's start, the stopping segment replayed with the sequential
arithmetic) and the algorithm the split forward kernels run
(`_kernel_split_forward`: k_forward's exact head, k_forward_chunk's chunks of
512 with the head's transmittance bounding their start, k_forward_replay's
replay on T_in times the running product, and the assembly).

Every step is float32 in the oracle's operation order, vectorised over a
tile's 256 pixels.  The model reproduces the oracle bit for bit when it does
not split.  Split, it must stay within the forward tolerance, and last_contrib
may differ only at pixels whose stop decision the oracle flags as a
knife-edge: the merged products round differently from the sequential ones.
"""
import numpy as np
import pytest

import gen
import oracle

F = np.float32
T_MIN, A_MIN, A_MAX, S_SKIP = F(1e-4), F(1.0) / F(255.0), F(0.999), F(5.55)
EPS_ALPHA = 6e-7       # the GPU parity margins: sigma in the same order, exp within a few ulp


def _alpha(s, px, py):
    """alpha of splat s at the pixels, and whether it passes the skips."""
    dx = px - s[0]
    dy = py - s[1]
    sigma = F(0.5) * (s[2] * dx * dx + s[4] * dy * dy) + s[3] * dx * dy
    e = np.exp(-sigma.astype(np.float64)).astype(F)
    raw = s[8] * e
    alpha = np.where(raw < A_MAX, raw, A_MAX).astype(F)
    ok = (sigma >= F(0)) & (sigma < S_SKIP) & (alpha >= A_MIN)
    return alpha, ok


def _sequential(splats, lst, pos0, px, py, C, T, last, done):
    """The per-pixel forward over lst (positions pos0, pos0 + 1, ...) from the
    given state, with the stop; updates the state in place."""
    for k, i in enumerate(lst):
        if done.all():
            break
        s = splats[i]
        alpha, ok = _alpha(s, px, py)
        ok &= ~done
        next_t = (T * (F(1) - alpha)).astype(F)
        stop = ok & (next_t < T_MIN)
        comp = ok & ~stop
        w = (alpha * T).astype(F)
        for ch in range(3):
            C[ch] = np.where(comp, C[ch] + s[5 + ch] * w, C[ch]).astype(F)
        T[:] = np.where(comp, next_t, T)
        last[:] = np.where(comp, pos0 + k + 1, last)
        done |= stop


def _segment(splats, lst, px, py):
    """A segment from T = 1 without the stop: (C_k, P_k, last_k)."""
    C = np.zeros((3, px.size), F)
    P = np.ones(px.size, F)
    last = np.zeros(px.size, np.int64)
    for k, i in enumerate(lst):
        s = splats[i]
        alpha, ok = _alpha(s, px, py)
        w = (alpha * P).astype(F)
        for ch in range(3):
            C[ch] = np.where(ok, C[ch] + s[5 + ch] * w, C[ch]).astype(F)
        P = np.where(ok, (P * (F(1) - alpha)).astype(F), P)
        last = np.where(ok, k + 1, last)
    return C, P, last


def _split_forward(splats, lst, px, py, inside, seg_len, bounds=None):
    """The split forward; `bounds` (a list) receives the (T, C) state after
    each segment, the backward segments' starting points."""
    n = px.size
    C = np.zeros((3, n), F)
    T = np.ones(n, F)
    last = np.zeros(n, np.int64)
    done = ~inside
    replays = 0
    for lo in range(0, len(lst), seg_len):
        seg = lst[lo:lo + seg_len]
        Ck, Pk, lk = _segment(splats, seg, px, py)
        prod = (T * Pk).astype(F)
        merge = ~done & (prod >= T_MIN)
        for ch in range(3):
            C[ch] = np.where(merge, C[ch] + (T * Ck[ch]).astype(F), C[ch]).astype(F)
        last = np.where(merge & (lk > 0), lo + lk, last)
        T = np.where(merge, prod, T)
        replay = ~done & ~merge
        if replay.any():
            replays += int(replay.sum())
            sub_done = ~replay
            _sequential(splats, seg, lo, px, py, C, T, last, sub_done)
            done |= replay & sub_done
        if bounds is not None:
            bounds.append((T.copy(), C.copy()))
    return C, T, last, replays


def _kernel_split_forward(splats, lst, px, py, inside, head, chunk=512):
    """The split forward as its kernels compute it, for one tile whose list
    is longer than `head` (a multiple of `chunk`): returns (C, T, last, the
    stop chunk per pixel or -1)."""
    n = px.size
    # k_forward: the exact head
    C = np.zeros((3, n), F)
    T = np.ones(n, F)
    last = np.zeros(n, np.int64)
    done = ~inside
    _sequential(splats, lst[:head], 0, px, py, C, T, last, done)
    t_head = T.copy()
    nchunks = (len(lst) + chunk - 1) // chunk
    first = head // chunk
    # k_forward_chunk: every chunk past the head from T = 1, a pixel leaving
    # once t_head times its product falls below the threshold
    Ck, Pk, Lk = [], [], []
    for k in range(first, nchunks):
        seg = lst[k * chunk:(k + 1) * chunk]
        c = np.zeros((3, n), F)
        P = np.ones(n, F)
        lk = np.zeros(n, np.int64)
        gone = done.copy()
        for j, i in enumerate(seg):
            s = splats[i]
            alpha, ok = _alpha(s, px, py)
            ok &= ~gone
            nxt = (P * (F(1) - alpha)).astype(F)
            stop = ok & ((t_head * nxt).astype(F) < T_MIN)
            comp = ok & ~stop
            w = (alpha * P).astype(F)
            for ch in range(3):
                c[ch] = np.where(comp, c[ch] + s[5 + ch] * w, c[ch]).astype(F)
            P = np.where(comp | stop, nxt, P)
            lk = np.where(comp, j + 1, lk)
            gone |= stop
        Ck.append(c)
        Pk.append(P)
        Lk.append(lk)
    # the chunks' prepare: the first chunk at whose end the product chain
    # falls below the threshold holds the stop
    stop_chunk = np.full(n, -1, np.int64)
    T_at = np.zeros((nchunks - first, n), F)
    Tr = t_head.copy()
    live = ~done
    for q, k in enumerate(range(first, nchunks)):
        T_at[q] = Tr
        Tn = (Tr * Pk[q]).astype(F)
        st = live & (Tn < T_MIN)
        stop_chunk = np.where(st, k, stop_chunk)
        adv = live & ~st
        for ch in range(3):
            C[ch] = np.where(adv, C[ch] + (Tr * Ck[q][ch]).astype(F), C[ch]).astype(F)
        last = np.where(adv & (Lk[q] > 0), k * chunk + Lk[q], last)
        Tr = np.where(adv, Tn, Tr)
        live &= ~st
    T = np.where(~done, Tr, T)
    # k_forward_replay: the stopping chunk from its start transmittance, on
    # t_in times the running product
    for k in np.unique(stop_chunk[stop_chunk >= 0]):
        mine = stop_chunk == k
        t_in = T_at[k - first]
        seg = lst[k * chunk:(k + 1) * chunk]
        c = np.zeros((3, n), F)
        P = np.ones(n, F)
        lr = np.zeros(n, np.int64)
        gone = ~mine
        for j, i in enumerate(seg):
            s = splats[i]
            alpha, ok = _alpha(s, px, py)
            ok &= ~gone
            nxt = (P * (F(1) - alpha)).astype(F)
            stop = ok & ((t_in * nxt).astype(F) < T_MIN)
            comp = ok & ~stop
            w = (alpha * P).astype(F)
            for ch in range(3):
                c[ch] = np.where(comp, c[ch] + s[5 + ch] * w, c[ch]).astype(F)
            P = np.where(comp, nxt, P)
            lr = np.where(comp, j + 1, lr)
            gone |= stop
        assert gone[mine].all(), "a replay must stop inside its chunk"
        for ch in range(3):
            C[ch] = np.where(mine, C[ch] + (t_in * c[ch]).astype(F), C[ch]).astype(F)
        T = np.where(mine, (t_in * P).astype(F), T)
        last = np.where(mine & (lr > 0), k * chunk + lr, last)
    return C, T, last, stop_chunk


def _heavy_tiles(ranges, count):
    lengths = ranges[:, 1].astype(np.int64) - ranges[:, 0].astype(np.int64)
    return np.argsort(-lengths, kind="stable")[:count]


@pytest.fixture(scope="module")
def lego_final():
    wl = gen.lego_final()
    _, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    ranges = ranges.reshape(-1, 2)
    f = oracle.forward(wl.splats, idx, ranges, wl.width, wl.height, eps_alpha=EPS_ALPHA, sigma_ulps=0.0)
    return wl, idx, ranges, f


def _tile_pixels(wl, tile):
    tiles_x = (wl.width + 15) // 16
    x0, y0 = (tile % tiles_x) * 16, (tile // tiles_x) * 16
    y, x = np.divmod(np.arange(256), 16)
    x, y = x0 + x, y0 + y
    inside = (x < wl.width) & (y < wl.height)
    p = np.where(inside, y * wl.width + x, 0)
    return x.astype(F), y.astype(F), inside, p


def test_unsplit_model_is_the_oracle(lego_final):
    wl, idx, ranges, f = lego_final
    splats = wl.splats.astype(F)
    tile = int(_heavy_tiles(ranges, 1)[0])
    px, py, inside, p = _tile_pixels(wl, tile)
    lst = idx[ranges[tile, 0]:ranges[tile, 1]]
    C, T, last = np.zeros((3, 256), F), np.ones(256, F), np.zeros(256, np.int64)
    _sequential(splats, lst, 0, px, py, C, T, last, ~inside)
    assert np.array_equal(C.T[inside], f["out"][p[inside], :3])
    assert np.array_equal(T[inside], f["final_T"][p[inside]])
    assert np.array_equal(last[inside], f["last"][p[inside]].astype(np.int64))


@pytest.mark.parametrize("seg_len", [512, 300])
def test_split_forward_matches_the_oracle(lego_final, seg_len):
    """The four longest lists of the Lego-final set, cut into segments."""
    wl, idx, ranges, f = lego_final
    splats = wl.splats.astype(F)
    total_replays = 0
    for tile in _heavy_tiles(ranges, 4):
        tile = int(tile)
        px, py, inside, p = _tile_pixels(wl, tile)
        lst = idx[ranges[tile, 0]:ranges[tile, 1]]
        assert len(lst) > 2 * seg_len
        C, T, last, replays = _split_forward(splats, lst, px, py, inside, seg_len)
        total_replays += replays
        ref_c, ref_t = f["out"][p, :3], f["final_T"][p]
        d = np.maximum(np.abs(C.T - ref_c).max(axis=1), np.abs(T - ref_t))
        knife = f["margin"][p] < 1.0
        bad = inside & ((d > 1e-5) | (last != f["last"][p].astype(np.int64)))
        assert not (bad & ~knife).any(), (tile, np.nonzero(bad & ~knife)[0][:5])
        assert d[inside & ~knife].max() <= 1e-5
    assert total_replays > 0    # the stop fell inside a segment somewhere


@pytest.mark.parametrize("name,tiles", [("lego_far", 3), ("lego_final", 2)])
def test_kernel_split_forward_matches_the_oracle(name, tiles):
    """The split forward's algorithm with a 1,024-position head and 512-position
    chunks on the longest lists of the crowded close-up and of the Lego-final
    set: within the forward tolerance of the oracle, last_contrib moved only at
    knife-edges, and the replays always find the stop inside their chunk."""
    wl = gen.make(name)
    _, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    ranges = ranges.reshape(-1, 2)
    f = oracle.forward(wl.splats, idx, ranges, wl.width, wl.height, eps_alpha=EPS_ALPHA, sigma_ulps=0.0)
    splats = wl.splats.astype(F)
    stops = 0
    for tile in _heavy_tiles(ranges, tiles):
        tile = int(tile)
        px, py, inside, p = _tile_pixels(wl, tile)
        lst = idx[ranges[tile, 0]:ranges[tile, 1]]
        assert len(lst) > 1024 + 512
        C, T, last, stop_chunk = _kernel_split_forward(splats, lst, px, py, inside, 1024)
        stops += int((stop_chunk >= 0).sum())
        ref_c, ref_t = f["out"][p, :3], f["final_T"][p]
        d = np.maximum(np.abs(C.T - ref_c).max(axis=1), np.abs(T - ref_t))
        knife = f["margin"][p] < 1.0
        bad = inside & ((d > 1e-5) | (last != f["last"][p].astype(np.int64)))
        assert not (bad & ~knife).any(), (tile, np.nonzero(bad & ~knife)[0][:5])
        assert d[inside & ~knife].max() <= 1e-5
    assert stops > 0    # some pixels stop past their head, inside a chunk


# --- backward ------------------------------------------------------------------

def _backward_segment(splats, lst, lo, px, py, g, L, T, S, acc):
    """Back to front over positions lo + k of one segment, from the state at its
    end: T (transmittance behind it) and S (colour composited behind it).  The
    per-pixel backward's formulas, with T un-blended as T / (1 - alpha); the
    per-splat sums go to acc (float64)."""
    T, S = T.copy(), S.copy()
    for k in range(len(lst) - 1, -1, -1):
        i = lst[k]
        s = splats[i]
        dx = px - s[0]
        dy = py - s[1]
        sigma = F(0.5) * (s[2] * dx * dx + s[4] * dy * dy) + s[3] * dx * dy
        e = np.exp(-sigma.astype(np.float64)).astype(F)
        raw = (s[8] * e).astype(F)
        alpha = np.where(raw < A_MAX, raw, A_MAX).astype(F)
        comp = (lo + k < L) & (sigma >= F(0)) & (sigma < S_SKIP) & (alpha >= A_MIN)
        if not comp.any():
            continue
        one_m = (F(1) - alpha).astype(F)
        tj = (T / one_m).astype(F)
        at = (alpha * tj).astype(F)
        da = sum(g[ch] * (s[5 + ch] * tj - S[ch] / one_m) for ch in range(3)).astype(F)
        draw = np.where(comp & (raw < A_MAX), da, F(0)).astype(F)
        dsig = (-draw * raw).astype(F)
        v = [-dsig * (s[2] * dx + s[3] * dy), -dsig * (s[3] * dx + s[4] * dy), dsig * (F(0.5) * dx * dx),
             dsig * (dx * dy), dsig * (F(0.5) * dy * dy)]
        v += [np.where(comp, g[ch] * at, F(0)) for ch in range(3)] + [draw * e]
        acc[i] += [float(np.sum(x[comp], dtype=np.float64)) for x in v]
        for ch in range(3):
            S[ch] = np.where(comp, S[ch] + s[5 + ch] * at, S[ch]).astype(F)
        T = np.where(comp, tj, T)


def _overlap_set(seed=5):
    """48x32 px (6 tiles), 2,500 splats of 3 to 12 px std over the frame, at
    opacities 0.005 to 0.06: every list is about 2,000 long and nearly all of
    it is composited; 95 pixels stop near its end, the others never do."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n, w, h = 2500, 48, 32
    sp = np.zeros((n, 9), np.float32)
    sp[:, 0] = rng.uniform(-8, w + 8, n)
    sp[:, 1] = rng.uniform(-8, h + 8, n)
    std = rng.uniform(3.0, 12.0, n)
    rho = rng.uniform(-0.5, 0.5, n)
    sp[:, 2] = 1.0 / (std ** 2 * (1 - rho ** 2))
    sp[:, 3] = -rho / (std ** 2 * (1 - rho ** 2))
    sp[:, 4] = 1.0 / (std ** 2 * (1 - rho ** 2))
    sp[:, 5:8] = rng.uniform(0, 1, (n, 3))
    sp[:, 8] = rng.uniform(0.005, 0.06, n)
    return gen.from_arrays("split_overlap", w, h, sp, rng.uniform(1, 9, n).astype(np.float32), seed=seed)


@pytest.mark.parametrize("seg_len", [None, 256])
def test_split_backward_matches_the_oracle(seg_len):
    """Gradients of the whole frame from per-tile segments (None: one segment
    per tile, the per-pixel kernel's scheme), each started from the forward's
    boundary state, against the oracle within the GPU parity tolerance."""
    wl = _overlap_set()
    splats = wl.splats.astype(F)
    _, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    ranges = ranges.reshape(-1, 2)
    o = oracle.backward(wl.splats, idx, ranges, wl.width, wl.height, wl.dl_dout, eps_alpha=EPS_ALPHA,
                        sigma_ulps=0.0)
    f = oracle.forward(wl.splats, idx, ranges, wl.width, wl.height, eps_alpha=EPS_ALPHA, sigma_ulps=0.0)
    acc = np.zeros((wl.n, 9))
    segments = 0
    for tile in range(len(ranges)):
        lst = idx[ranges[tile, 0]:ranges[tile, 1]]
        px, py, inside, p = _tile_pixels(wl, tile)
        g = np.where(inside, wl.dl_dout[p, :3].T, F(0)).astype(F)
        L = np.where(inside, f["last"][p].astype(np.int64), 0)
        seg = seg_len or max(len(lst), 1)
        bounds = []
        C, T, last, _ = _split_forward(splats, lst, px, py, inside, seg, bounds)
        assert np.array_equal(last[inside], L[inside])
        for k, lo in enumerate(range(0, len(lst), seg)):
            tb, cb = bounds[k]
            _backward_segment(splats, lst[lo:lo + seg], lo, px, py, g, L, tb, (C - cb).astype(F), acc)
            segments += 1
    ref = o["grad"]
    tol = 1e-4 + 1e-4 * np.abs(ref) + 8 * 2.0 ** -24 * o["gabs"]
    bad = np.any(np.abs(acc - ref) > tol, axis=1) & ~o["knife"]
    assert not bad.any(), np.nonzero(bad)[0][:5]
    assert segments >= (6 if seg_len is None else 40)
    assert np.abs(ref).max() > 1.0      # the gradients are not vacuous
    assert f["last"].min() > 6 * 256    # every segment holds composited splats
    assert 0 < int((f["final_T"] < 1.1e-4).sum()) < wl.width * wl.height   # some pixels stop
