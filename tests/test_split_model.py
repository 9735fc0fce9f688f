"""A CPU model of the heavy-tile split of the forward (not a kernel yet),
against the oracle.

Splitting one tile's list across CTAs ("next" row 3: several CTAs per long
list, merged through the (C, T) state) has to keep the early stop
(T < 1e-4).  A segment cannot know the transmittance in front of it, so the
model's segments composite from T = 1 without stopping and record their colour
C_k, their transmittance product P_k and their last composite.  A merge then
walks each pixel's segments in order.  While T_in P_k stays at or above 1e-4,
no stop can fall inside segment k (the running product only decreases), so
(C, T) <- (C + T_in C_k, T_in P_k).  Otherwise the pixel stops inside segment
k, and the merge replays that segment from (T_in, C) with the sequential
arithmetic.

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


def _split_forward(splats, lst, px, py, inside, seg_len):
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
    return C, T, last, replays


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
