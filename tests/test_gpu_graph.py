"""The forward and backward take no host synchronisation and allocate nothing
after their first call, so a caller can capture them in a CUDA graph: replays
give the same bits as direct calls (deterministic accumulation), and the graph
picks up new gradients of the loss written into its input buffer."""
import numpy as np
import pytest
import torch

import gen
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


def test_forward_backward_replay_in_a_graph(gsr):
    ctx = gsr.Context(0)
    try:
        ctx.set_option("deterministic", True)
        wl = gen.lego_early()
        sp, dp, dl = to_dev(wl.splats), to_dev(wl.depths), to_dev(wl.dl_dout)
        bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        npx = wl.width * wl.height
        out = torch.empty((npx, 4), dtype=torch.float32, device="cuda:0")
        fT = torch.empty((npx,), dtype=torch.float32, device="cuda:0")
        last = torch.empty((npx,), dtype=torch.int32, device="cuda:0")
        grad = torch.empty((wl.n, 9), dtype=torch.float32, device="cuda:0")

        def step():
            gsr.rasterize_forward(ctx, sp, bins, out, fT, last)
            gsr.rasterize_backward(ctx, sp, bins, dl, fT, last, grad)

        step()   # first call: the backward's buffers are allocated here
        torch.cuda.synchronize()
        ref_out, ref_grad = out.clone(), grad.clone()
        dl2 = to_dev(np.ascontiguousarray(wl.dl_dout[::-1]))
        step_in = dl.clone()
        dl.copy_(dl2)
        step()
        torch.cuda.synchronize()
        ref_grad2 = grad.clone()
        dl.copy_(step_in)

        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                step()
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(3):
            out.zero_()
            grad.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, ref_out)
            assert torch.equal(grad.view(torch.int32), ref_grad.view(torch.int32))
        dl.copy_(dl2)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(grad.view(torch.int32), ref_grad2.view(torch.int32))
    finally:
        ctx.close()
