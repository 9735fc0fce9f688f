"""Binning without a host read-back (gsr_reserve_pairs).

With a reservation the binning keeps its pair count on the device: every
kernel takes its key counts from there and the radix passes decide on the
device which digits to skip.  The results must be the same bits as the
default mode's and the oracle's; a count beyond the reservation must leave
empty bins and report itself; and the whole step (binning, forward, backward)
must replay from one CUDA graph with the same bits.
"""
import numpy as np
import pytest
import torch

import gen
from gpu_helpers import check_backward, check_bins, check_forward, run_gpu, run_oracle, to_dev

GSR_TOO_MANY_PAIRS = 4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


def _sync_free_ctx(gsr, reserve):
    ctx = gsr.Context(0)
    ctx.reserve_pairs(reserve)
    return ctx


@pytest.mark.parametrize("name", ["tiny", "small", "lego_early", "stress"])
def test_parity_without_read_back(gsr, name):
    wl = gen.make(name)
    ctx = _sync_free_ctx(gsr, 1 << 25)         # stress emits 23.6M pairs
    try:
        g = run_gpu(gsr, ctx, wl)
        o = run_oracle(wl)
        check_bins(g, o)
        check_forward(g, o)
        check_backward(g, o)
        st = ctx.bin_stats()
        assert st["num_pairs"] == len(o["keys"]) and st["capacity"] >= len(o["keys"])
    finally:
        ctx.close()


def _edge_cases():
    rng = np.random.default_rng(5)
    one = gen.from_arrays("one", 40, 30, np.array([[20, 15, 0.05, 0.01, 0.04, 0.3, 0.6, 0.9, 0.7]]), [2.0])
    n = 300
    sp = np.zeros((n, 9), np.float32)
    sp[:, 0:2] = rng.uniform(0, 16, (n, 2))
    sp[:, 2] = sp[:, 4] = 0.1
    sp[:, 5:8] = rng.uniform(0, 1, (n, 3))
    sp[:, 8] = rng.uniform(0.05, 0.9, n)
    one_tile_ties = gen.from_arrays("one_tile_ties", 16, 16, sp, np.full(n, 3.0, np.float32))  # no digit varies
    empty = gen.from_arrays("empty", 64, 48, np.zeros((0, 9), np.float32), np.zeros(0, np.float32))
    culled = gen.from_arrays("culled", 64, 48, sp[:50], np.full(50, -1.0, np.float32))
    ragged = gen.small()
    ragged = gen.from_arrays("ragged", 257, 15, ragged.splats, ragged.depths, seed=2)
    return [one, one_tile_ties, empty, culled, ragged]


@pytest.mark.parametrize("wl", _edge_cases(), ids=lambda w: w.name)
def test_edge_cases_without_read_back(gsr, wl):
    ctx = _sync_free_ctx(gsr, 4096)
    try:
        g = run_gpu(gsr, ctx, wl)
        o = run_oracle(wl)
        check_bins(g, o)
        check_forward(g, o)
        check_backward(g, o)
    finally:
        ctx.close()


def _huge(n=100, side=1024):
    """n splats that each cover the whole side x side image: n x 4,096 pairs."""
    rng = np.random.default_rng(9)
    sp = np.zeros((n, 9), np.float32)
    sp[:, 0:2] = side / 2 + rng.uniform(-8, 8, (n, 2))
    sp[:, 2] = sp[:, 4] = 1.0 / (side * side)          # std = side px: the 3-sigma box covers the image
    sp[:, 5:8] = rng.uniform(0, 1, (n, 3))
    sp[:, 8] = rng.uniform(0.001, 0.01, n)
    return gen.from_arrays("huge", side, side, sp, rng.uniform(1, 5, n).astype(np.float32), seed=4)


def test_a_count_beyond_the_reservation_leaves_empty_bins(gsr):
    wl = _huge()                                   # 409,600 pairs > max(65536, 16 n)
    ctx = _sync_free_ctx(gsr, 1000)
    try:
        sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
        bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        with pytest.raises(gsr.GsrError) as err:
            ctx.num_pairs()
        assert err.value.code == GSR_TOO_MANY_PAIRS and "409600" in str(err.value)
        res = bins.raw.num_pairs_dev
        st = torch.as_tensor(gsr._abi._DeviceArray(res, (2,), "<i4"), device="cuda:0").cpu().numpy()
        assert st[0] == 409600 and st[1] == GSR_TOO_MANY_PAIRS
        assert not bins.tile_ranges().any()
        out, fT, last = gsr.rasterize_forward(ctx, sp, bins)
        grad = gsr.rasterize_backward(ctx, sp, bins, dl, fT, last)
        assert torch.all(fT == 1.0) and not out.any() and not last.any() and not grad.any()
        # with room for them the same call bins every pair
        ctx.reserve_pairs(500_000)
        g = run_gpu(gsr, ctx, wl)
        o = run_oracle(wl)
        check_bins(g, o)
        check_forward(g, o)
        check_backward(g, o)
    finally:
        ctx.close()


def test_read_back_and_reserved_modes_give_the_same_bits(gsr):
    wl = gen.lego_early()
    a, b = gsr.Context(0), _sync_free_ctx(gsr, 3_000_000)   # lego_early emits 2,320,479 pairs
    try:
        for c in (a, b):
            c.set_option("deterministic", True)
        ga, gb = run_gpu(gsr, a, wl), run_gpu(gsr, b, wl)
        for k in ("keys", "idx", "ranges", "out", "final_T", "last", "grad"):
            assert np.array_equal(ga[k].view(np.uint8), gb[k].view(np.uint8)), k
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("name,split_forward", [("lego_early", False), ("lego_far", True)])
def test_whole_step_replays_from_one_graph(gsr, name, split_forward):
    """Binning, forward and backward captured in one CUDA graph: the replays
    give the direct calls' bits, and pick up new inputs written in place
    (with the forward split too: its chunk queue lives on the device)."""
    wl = gen.make(name)
    ctx = _sync_free_ctx(gsr, 3_000_000)    # lego_early emits 2,320,479 pairs, lego_far 876,855
    try:
        ctx.set_option("deterministic", True)
        ctx.set_option("split_forward", split_forward)
        sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
        npx = wl.width * wl.height
        out = torch.empty((npx, 4), dtype=torch.float32, device="cuda:0")
        fT = torch.empty((npx,), dtype=torch.float32, device="cuda:0")
        last = torch.empty((npx,), dtype=torch.int32, device="cuda:0")
        grad = torch.empty((wl.n, 9), dtype=torch.float32, device="cuda:0")
        holder = {}

        def step():
            b = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
            gsr.rasterize_forward(ctx, sp, b, out, fT, last)
            gsr.rasterize_backward(ctx, sp, b, dl, fT, last, grad)
            holder["bins"] = b

        step()                      # allocations happen here, outside the capture
        torch.cuda.synchronize()
        ref = {"keys": holder["bins"].keys().clone(), "out": out.clone(), "grad": grad.clone()}
        moved = sp.clone()
        moved[:, 0] += 3.0          # a second input: every splat 3 px to the right
        sp_saved = sp.clone()
        sp.copy_(moved)
        step()
        torch.cuda.synchronize()
        ref2 = {"out": out.clone(), "grad": grad.clone()}
        sp.copy_(sp_saved)

        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                step()
        torch.cuda.current_stream().wait_stream(s)
        launches = ctx.launch_count()
        for _ in range(3):
            out.zero_()
            grad.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(holder["bins"].keys(), ref["keys"])
            assert torch.equal(out, ref["out"])
            assert torch.equal(grad.view(torch.int32), ref["grad"].view(torch.int32))
        assert ctx.launch_count() == launches      # replays launch through the graph only
        sp.copy_(moved)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref2["out"])
        assert torch.equal(grad.view(torch.int32), ref2["grad"].view(torch.int32))
    finally:
        ctx.close()
