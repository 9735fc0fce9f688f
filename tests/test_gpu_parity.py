"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Binning must match bit for bit (sorted keys, sorted indices, tile ranges);
forward pixels within 1e-5 absolute with last_contrib equal; gradients within
1e-4 + 1e-4 |ref| (+ 8u sum|t| for sums whose terms cancel, on at most a stated
number of components per config).  A threshold decision (alpha vs 1/255, T vs
1e-4, the 0.999 clamp) whose tested value lies within the two sides' rounding
uncertainty may go either way; a pixel or splat passes then only if the oracle,
re-run with such decisions taken the other way, reproduces the GPU within the
same tolerances.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
from gpu_helpers import (check_backward, check_bins, check_forward, record_stats, run_gpu, run_oracle, to_dev,
                         varying_digit_mask)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


@pytest.fixture(scope="module")
def ctx(gsr):
    c = gsr.Context(0)
    yield c
    c.close()


# The most gradient components per config allowed to need the 8u sum|t| term
# (sums whose terms cancel), with the forced replays applied.  Measured on
# GB300: tiny 0, small 0, lego_early 2 (of 0.75M), lego_final 0 (of 3.7M),
# stress 24 (of 9M); the caps leave room for the order of the atomic adds.
COND_CAPS = {"tiny": 0, "small": 0, "lego_early": 4, "lego_final": 2, "stress": 32}


def _full(gsr, ctx, wl, backward=True, cond_cap=None):
    g = run_gpu(gsr, ctx, wl, backward)
    o = run_oracle(wl, backward)
    check_bins(g, o)
    fs = check_forward(g, o)
    bs = check_backward(g, o, cond_cap=cond_cap) if backward else None
    record_stats(wl.name, pairs=int(g["num_pairs"]), forward=fs, backward=bs)
    return g, o, fs, bs


@pytest.mark.parametrize("name", ["tiny", "small", "lego_early", "lego_final"])
def test_config_parity(gsr, ctx, name):
    g, o, fs, bs = _full(gsr, ctx, gen.make(name), cond_cap=COND_CAPS[name])
    print(name, "pairs", g["num_pairs"], "forward", fs, "backward", bs)


def test_stress_parity(gsr, ctx):
    wl = gen.stress()
    g, o, fs, bs = _full(gsr, ctx, wl, cond_cap=COND_CAPS["stress"])
    print("stress pairs", g["num_pairs"], "forward", fs, "backward", bs)


@pytest.mark.parametrize("size", [32, 24])
def test_overlap_fixtures(gsr, ctx, size):
    _full(gsr, ctx, gen.overlap_fixture(size))


def test_elongated_parity(gsr, ctx):
    """Thin rotated splats of every size: the oriented culling of staged splats
    against pixel blocks must not drop an evaluation the oracle makes."""
    _full(gsr, ctx, gen.elongated_fixture())


def _random(n, w, h, seed, levels=None, big=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    s = np.zeros((n, 9), dtype=np.float32)
    s[:, 0] = rng.uniform(-20, w + 20, n)
    s[:, 1] = rng.uniform(-20, h + 20, n)
    std = rng.uniform(0.4, 10.0, n)
    if big:
        std[:big] = rng.uniform(max(w, h) * 0.5, max(w, h) * 2.0, big)
    s[:, 2] = 1.0 / std ** 2
    s[:, 3] = rng.uniform(-0.4, 0.4, n) / std ** 2
    s[:, 4] = 1.0 / std ** 2
    s[:, 5:8] = rng.uniform(0, 1, (n, 3))
    s[:, 8] = rng.uniform(0.0, 1.0, n)
    d = (rng.integers(1, levels + 1, n) if levels else rng.uniform(0.5, 30.0, n)).astype(np.float32)
    return gen.from_arrays(f"rand{n}", w, h, s, d, seed=seed + 100)


@pytest.mark.parametrize("n", [0, 1, 255, 256, 257, 1234])
def test_sizes(gsr, ctx, n):
    _full(gsr, ctx, _random(n, 96, 80, n))


def test_tie_heavy_depths(gsr, ctx):
    # 8 distinct depths over 5000 splats: equal keys must come out in splat order.
    _full(gsr, ctx, _random(5000, 128, 128, 9, levels=8))


@pytest.mark.parametrize("w,h", [(100, 70), (1, 1), (17, 33), (16, 16), (257, 15)])
def test_ragged_images(gsr, ctx, w, h):
    _full(gsr, ctx, _random(600, w, h, w * 1000 + h))


def test_maximum_image_side(gsr, ctx):
    """The widest image the API takes (2^19 px, 32768 tiles in a row): tile
    coordinates at the top of their 16-bit packing, 15-bit tile ids, splats
    over both ends of the strip."""
    w, h, n = 1 << 19, 16, 64
    rng = np.random.Generator(np.random.PCG64(11))
    s = np.zeros((n, 9), dtype=np.float32)
    s[:, 0] = np.concatenate([rng.uniform(-20, 60, 16), rng.uniform(w - 60, w + 20, 16), rng.uniform(0, w, 32)])
    s[:, 1] = rng.uniform(-4, h + 4, n)
    std = rng.uniform(0.5, 6.0, n)
    s[:, 2] = 1.0 / std ** 2
    s[:, 3] = rng.uniform(-0.3, 0.3, n) / std ** 2
    s[:, 4] = 1.0 / std ** 2
    s[:, 5:8] = rng.uniform(0, 1, (n, 3))
    s[:, 8] = rng.uniform(0.05, 1.0, n)
    d = rng.uniform(0.5, 20.0, n).astype(np.float32)
    g, o, fs, bs = _full(gsr, ctx, gen.from_arrays("max_side", w, h, s, d, seed=12))
    assert int(o["keys"].max() >> 32) == (w // 16) - 1  # a splat reaches the last tile


def test_huge_splats_long_lists(gsr, ctx):
    # A few splats cover every tile; every tile list holds thousands of entries.
    _full(gsr, ctx, _random(3000, 160, 144, 5, big=40))


def test_culled_splats(gsr, ctx):
    wl = _random(400, 64, 64, 3)
    s, d = wl.splats, wl.depths
    s[0, 2] = -1.0                  # a <= 0
    s[1, 3] = 10.0                  # indefinite (det <= 0)
    d[2] = 0.0                      # depth 0
    d[3] = -1.0                     # behind
    s[4, 0] = np.nan                # non-finite field
    s[5, 8] = np.inf
    d[6] = np.inf
    s[7, 0:2] = [-500.0, -500.0]    # off image
    g, o, _, _ = _full(gsr, ctx, wl)
    assert not np.isin(np.arange(8), g["idx"]).any()


def test_all_culled_and_empty(gsr, ctx):
    wl = _random(50, 48, 48, 4)
    wl.depths[:] = -1.0
    g = run_gpu(gsr, ctx, wl)
    assert g["num_pairs"] == 0
    assert np.all(g["ranges"] == 0)
    assert np.all(g["out"] == 0) and np.all(g["final_T"] == 1) and np.all(g["last"] == 0)
    assert np.all(g["grad"] == 0)
    g = run_gpu(gsr, ctx, _random(0, 40, 40, 0))
    assert g["num_pairs"] == 0 and g["grad"].shape == (0, 9)


def test_radix_pass_skip(gsr, ctx):
    """Digits every key shares are skipped ("C0 resident arena + C1 pass skip",
    section 2, C1); the stats report which ran."""
    wl = gen.lego_final()
    g = run_gpu(gsr, ctx, wl, backward=False)
    st = ctx.bin_stats()
    o = run_oracle(wl, backward=False)
    check_bins(g, o)
    # 2500 tiles: 12 tile bits, sorted as two 6-bit digits.
    assert (st["tile_digits"], st["tile_digit_bits"]) == (2, 6)
    assert st["depth_pass_mask"] == varying_digit_mask(o["keys"], 0, 32, 4)
    assert st["tile_pass_mask"] == varying_digit_mask(o["keys"], 32, 44, 2)
    assert not (st["depth_pass_mask"] >> 3) & 1      # depths in [2,6) share their top byte
    assert st["radix_passes"] == bin(st["depth_pass_mask"]).count("1") + bin(st["tile_pass_mask"]).count("1")
    assert st["emitting"] == len(np.unique(o["idx"]))


def test_stress_tile_digits(gsr, ctx):
    wl = gen.stress()
    run_gpu(gsr, ctx, wl, backward=False)
    st = ctx.bin_stats()
    # 120 x 68 = 8160 tiles: 13 tile bits as a 7-bit and a 6-bit digit.
    assert (st["tile_digits"], st["tile_digit_bits"]) == (2, 7)


def test_radix_sort_40000_tiles(gsr, ctx):
    """The pages' sort check at 40,000 tiles ("C0 resident arena + C1 pass
    skip", section 2, C1): about 200k keys against a plain stable sort (the
    oracle's), 16 tile bits sorted as two 8-bit digits, depths over several
    binades so that all four depth digits vary.  Binning only: a 3200x3200
    frame."""
    rng = np.random.Generator(np.random.PCG64(40_000))
    w = h = 3200
    n = 50_000
    s = np.zeros((n, 9), dtype=np.float32)
    s[:, 0] = rng.uniform(-10, w + 10, n)
    s[:, 1] = rng.uniform(-10, h + 10, n)
    std = rng.uniform(0.4, 5.0, n)
    s[:, 2] = 1.0 / std ** 2
    s[:, 3] = rng.uniform(-0.3, 0.3, n) / std ** 2
    s[:, 4] = 1.0 / std ** 2
    s[:, 5:9] = rng.uniform(0, 1, (n, 4))
    d = rng.uniform(0.5, 30.0, n).astype(np.float32)
    sp, dp = to_dev(s), to_dev(d)
    bins = gsr.bin_splats(ctx, sp, dp, w, h)
    g = {"keys": bins.keys().cpu().numpy().view(np.uint64), "idx": bins.sorted_idx().cpu().numpy().view(np.uint32),
         "ranges": bins.tile_ranges().cpu().numpy().view(np.uint32), "num_pairs": bins.num_pairs}
    st = ctx.bin_stats()
    keys, idx, ranges = oracle.bin_splats(s, d, w, h)
    check_bins(g, {"keys": keys, "idx": idx, "ranges": ranges})
    assert 150_000 < len(keys) < 400_000
    assert (st["tile_digits"], st["tile_digit_bits"]) == (2, 8)
    assert st["tile_pass_mask"] == varying_digit_mask(keys, 32, 48, 2) == 0b11
    assert st["depth_pass_mask"] == varying_digit_mask(keys, 0, 32, 4) == 0b1111


def test_no_pass_needed(gsr, ctx):
    # One tile, one depth: every digit is constant; the emitted order is the result.
    s = np.tile(np.array([[8.0, 8.0, 1.0, 0.0, 1.0, 0.5, 0.5, 0.5, 0.5]], np.float32), (300, 1))
    wl = gen.from_arrays("flat", 16, 16, s, np.full(300, 2.0, np.float32))
    g = run_gpu(gsr, ctx, wl)
    assert ctx.bin_stats()["radix_passes"] == 0
    o = run_oracle(wl)
    check_bins(g, o)
    check_forward(g, o)
    check_backward(g, o)


def test_arena_grows_and_reuses(gsr, ctx):
    caps = []
    for name in ["tiny", "lego_early", "small", "lego_early"]:
        wl = gen.make(name)
        g = run_gpu(gsr, ctx, wl, backward=False)
        check_bins(g, run_oracle(wl, backward=False))
        caps.append(ctx.bin_stats()["capacity"])
    assert caps == sorted(caps)          # grow-only
    assert caps[-1] == caps[1]           # reused, not regrown


def test_backward_variants_single_pixel_bit_equal(gsr, ctx):
    """dL/dout nonzero at one pixel: one nonzero term per splat, so every
    backward variant must give the same bits ("W1 warp sparse skip + exp-skip",
    section 1, parity (2))."""
    wl = gen.overlap_fixture(32)
    dl = np.zeros_like(wl.dl_dout)
    dl[15 * 32 + 17, :3] = [0.3, -1.2, 0.7]
    wl.dl_dout = dl
    results = []
    for skip in (1, 0):
        for lc in (1, 0):
            ctx.set_option("bwd_warp_skip", skip)
            ctx.set_option("bwd_last_contrib", lc)
            results.append(run_gpu(gsr, ctx, wl))
    ctx.set_option("bwd_warp_skip", 1)
    ctx.set_option("bwd_last_contrib", 1)
    for r in results[1:]:
        assert np.array_equal(r["grad"].view(np.uint32), results[0]["grad"].view(np.uint32))
    assert np.any(results[0]["grad"] != 0)
    check_backward(results[0], run_oracle(wl))


def test_backward_variants_agree(gsr, ctx):
    wl = gen.small()
    o = run_oracle(wl)
    for skip in (0, 1):
        for lc in (0, 1):
            ctx.set_option("bwd_warp_skip", skip)
            ctx.set_option("bwd_last_contrib", lc)
            check_backward(run_gpu(gsr, ctx, wl), o)
    ctx.set_option("bwd_warp_skip", 1)
    ctx.set_option("bwd_last_contrib", 1)


@pytest.mark.parametrize("name", ["lego_early", "stress", "elongated"])
def test_warp_culling_changes_nothing(gsr, ctx, name):
    """Warps skip splats whose alpha >= 1/255 ellipse misses their pixel block;
    the per-pixel tests would have skipped every one of those evaluations, so
    the forward must be bit-identical with culling off, and the backward
    identical up to the order of its double-precision sums."""
    wl = gen.elongated_fixture() if name == "elongated" else gen.make(name)
    on = run_gpu(gsr, ctx, wl)
    ctx.set_option("warp_cull", 0)
    try:
        off = run_gpu(gsr, ctx, wl)
    finally:
        ctx.set_option("warp_cull", 1)
    for k in ("out", "final_T", "last"):
        assert np.array_equal(on[k], off[k]), k
    assert np.allclose(on["grad"], off["grad"], rtol=1e-6, atol=1e-9)


def test_dependent_launch_changes_nothing(gsr, ctx):
    """Kernels launched with programmatic dependent launch wait for the grids
    before them, so the results are those of plain stream order."""
    wl = gen.lego_early()
    on = run_gpu(gsr, ctx, wl)
    ctx.set_option("pdl", 0)
    try:
        off = run_gpu(gsr, ctx, wl)
    finally:
        ctx.set_option("pdl", 1)
    for k in ("keys", "idx", "ranges", "out", "final_T", "last"):
        assert np.array_equal(on[k], off[k]), k
    assert np.allclose(on["grad"], off["grad"], rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("name", ["lego_final", "stress"])
def test_tile_order_is_a_longest_first_permutation(gsr, ctx, name):
    """bins.tile_order holds every tile once, longest lists first: a tile may
    precede a longer one only within the 2^(1/8) width of a cost class."""
    wl = gen.make(name)
    sp, dp = to_dev(wl.splats), to_dev(wl.depths)
    bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
    order = bins.tile_order().cpu().numpy().view(np.uint32).astype(np.int64)
    r = bins.tile_ranges().cpu().numpy().view(np.uint32).astype(np.int64)
    lengths = (r[:, 1] - r[:, 0])[order]
    assert np.array_equal(np.sort(order), np.arange(len(r)))
    later_max = np.maximum.accumulate(lengths[::-1])[::-1]   # longest list at or after each position
    assert np.all(later_max <= np.maximum(lengths * 2 ** 0.25, lengths + 1)), "a much longer tile comes later"


def test_results_do_not_depend_on_tile_order(gsr, ctx):
    """Bins without a launch order (NULL, e.g. built by a caller) give the same
    forward bit for bit and the same gradients up to the order of their sums."""
    wl = gen.lego_early()
    sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
    bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
    out_a, t_a, l_a = [x.clone() for x in gsr.rasterize_forward(ctx, sp, bins)]
    g_a = gsr.rasterize_backward(ctx, sp, bins, dl, t_a, l_a).clone()
    bins.raw.tile_order = None
    out_b, t_b, l_b = gsr.rasterize_forward(ctx, sp, bins)
    torch.cuda.synchronize()
    for a, b in ((out_a, out_b), (t_a, t_b), (l_a, l_b)):
        assert torch.equal(a, b)
    g_b = gsr.rasterize_backward(ctx, sp, bins, dl, t_b, l_b)
    assert np.allclose(g_a.cpu().numpy(), g_b.cpu().numpy(), rtol=1e-6, atol=1e-9)


def test_self_noise(gsr, ctx):
    """Run-to-run spread of the atomically accumulated gradients (the pages'
    self-noise protocol: 20 repeats, "M3 per-splat backward", section 2)."""
    wl = gen.small()
    sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
    bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
    out, t, last = gsr.rasterize_forward(ctx, sp, bins)
    runs = [gsr.rasterize_backward(ctx, sp, bins, dl, t, last).cpu().numpy().astype(np.float64)
            for _ in range(20)]
    ref = runs[0]
    # Spread in units of the parity tolerance (1e-4 + 1e-4 |g|): atomics may
    # reorder the sums but must stay far inside it.
    worst = max(float(np.max(np.abs(r - ref) / (1e-4 + 1e-4 * np.abs(ref)))) for r in runs[1:])
    max_rel = max(float(np.max(np.abs(r - ref) / np.maximum(np.abs(ref), 1e-6))) for r in runs[1:])
    print("self-noise: max |d| / tolerance", worst, "max_rel", max_rel)
    assert worst < 0.1


def test_forward_deterministic(gsr, ctx):
    wl = gen.lego_early()
    a = run_gpu(gsr, ctx, wl, backward=False)
    b = run_gpu(gsr, ctx, wl, backward=False)
    for k in ("keys", "idx", "ranges", "out", "final_T", "last"):
        assert np.array_equal(a[k], b[k]), k


def test_invalid_arguments(gsr, ctx):
    dev = "cuda:0"
    sp = torch.zeros((4, 9), dtype=torch.float32, device=dev)
    dp = torch.ones(4, dtype=torch.float32, device=dev)
    with pytest.raises(gsr.GsrError) as e:
        gsr.bin_splats(ctx, sp, dp, 0, 16)
    assert e.value.code == 1
    with pytest.raises(gsr.GsrError):
        gsr.bin_splats(ctx, sp, dp, 16, (1 << 19) + 1)
    bins = gsr.bin_splats(ctx, sp, dp, 16, 16)
    with pytest.raises(gsr.GsrError):   # n differs from the bins'
        gsr.rasterize_forward(ctx, sp[:3], bins)
    base = torch.zeros(256 * 4 + 1, dtype=torch.float32, device=dev)
    misaligned = base[1:].view(256, 4)
    with pytest.raises(gsr.GsrError) as e:
        gsr.rasterize_forward(ctx, sp, bins, out_rgbw=misaligned)
    assert e.value.code == 1
    with pytest.raises(ValueError):
        gsr.bin_splats(ctx, sp.double(), dp, 16, 16)


def test_launch_count(gsr, ctx):
    wl = gen.tiny()
    before = ctx.launch_count()
    run_gpu(gsr, ctx, wl)
    assert ctx.launch_count() > before + 5
