"""Parity of the CUDA projection (forward and backward, through the C ABI) with
the double oracle, with the tolerances derived in tests/proj_checks.py; and the
whole chain projection -> binning -> forward -> backward -> projection backward
against the oracle chain."""
import numpy as np
import pytest
import torch

import gen
import oracle
import proj_checks
from gpu_helpers import GRAD_ATOL, GRAD_COND, GRAD_RTOL, run_gpu, run_oracle, to_dev

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


def _project(gsr, ctx, g32, cam, G32=None):
    g = to_dev(g32)
    sp, d = gsr.project_forward(ctx, g, cam)
    grad = None
    if G32 is not None:
        grad = gsr.project_backward(ctx, g, cam, to_dev(G32)).cpu().numpy()
    torch.cuda.synchronize()
    return sp.cpu().numpy(), d.cpu().numpy(), grad


@pytest.mark.parametrize("n", [1, 255, 256, 257, 5000])
def test_projection_parity_sizes(gsr, ctx, n):
    sc = gen.lego_scene(n=n, seed=40 + n)
    sp, d, grad = _project(gsr, ctx, sc.gaussians, sc.camera, sc.dl_dsplat)
    fs = proj_checks.check_forward(sc.gaussians, sc.camera, sp, d)
    bs = proj_checks.check_backward(sc.gaussians, sc.camera, sc.dl_dsplat, grad)
    print(n, fs, bs)


def test_projection_parity_lego_full(gsr, ctx):
    """All 409,660 Gaussians of the Lego-shaped scene, in the launch the bench times."""
    sc = gen.lego_scene()
    sp, d, grad = _project(gsr, ctx, sc.gaussians, sc.camera, sc.dl_dsplat)
    fs = proj_checks.check_forward(sc.gaussians, sc.camera, sp, d)
    bs = proj_checks.check_backward(sc.gaussians, sc.camera, sc.dl_dsplat, grad)
    print("lego", fs, bs)


def test_projection_edge_cases(gsr, ctx):
    """Behind the camera, inside the near plane, zero quaternion, NaN and inf
    fields (not visible: zeros, rgb copied, no gradient); needle-thin, very
    large and off-screen Gaussians (visible)."""
    e = gen.edge_scene()
    sp, d, grad = _project(gsr, ctx, e.gaussians, e.camera, e.dl_dsplat)
    fs = proj_checks.check_forward(e.gaussians, e.camera, sp, d)
    assert fs["invisible"] == 5 * 16
    proj_checks.check_backward(e.gaussians, e.camera, e.dl_dsplat, grad)


def test_projection_without_dilation(gsr, ctx):
    sc = gen.lego_scene(n=3000, seed=5)
    cam = sc.camera.copy()
    cam[17] = 0.0
    sp, d, grad = _project(gsr, ctx, sc.gaussians, cam, sc.dl_dsplat)
    proj_checks.check_forward(sc.gaussians, cam, sp, d)
    proj_checks.check_backward(sc.gaussians, cam, sc.dl_dsplat, grad)


def test_unaligned_arrays_give_the_same_bits(gsr, ctx):
    """Arrays that are not 16-byte aligned take the scalar staging path."""
    sc = gen.lego_scene(n=1000, seed=6)
    n = sc.n
    ref_sp, ref_d, ref_g = _project(gsr, ctx, sc.gaussians, sc.camera, sc.dl_dsplat)
    gbuf = torch.zeros(n * 14 + 1, dtype=torch.float32, device="cuda:0")
    gbuf[1:] = to_dev(sc.gaussians).reshape(-1)
    g = gbuf[1:].view(n, 14)
    spbuf = torch.zeros(n * 9 + 1, dtype=torch.float32, device="cuda:0")
    sp = spbuf[1:].view(n, 9)
    dbuf = torch.zeros(n + 1, dtype=torch.float32, device="cuda:0")
    gsr.project_forward(ctx, g, sc.camera, splats=sp, depths=dbuf[1:])
    Gbuf = torch.zeros(n * 9 + 1, dtype=torch.float32, device="cuda:0")
    Gbuf[1:] = to_dev(sc.dl_dsplat).reshape(-1)
    obuf = torch.zeros(n * 14 + 1, dtype=torch.float32, device="cuda:0")
    gsr.project_backward(ctx, g, sc.camera, Gbuf[1:].view(n, 9), dl_dgauss=obuf[1:].view(n, 14))
    assert np.array_equal(sp.cpu().numpy(), ref_sp)
    assert np.array_equal(dbuf[1:].cpu().numpy(), ref_d)
    assert np.array_equal(obuf[1:].view(n, 14).cpu().numpy(), ref_g)


def test_projection_empty_and_invalid(gsr, ctx):
    cam = gen.lego_scene(n=1).camera
    empty = torch.empty((0, 14), dtype=torch.float32, device="cuda:0")
    before = ctx.launch_count()
    sp, d = gsr.project_forward(ctx, empty, cam)
    assert sp.shape == (0, 9) and d.shape == (0,)
    gsr.project_backward(ctx, empty, cam, torch.empty((0, 9), dtype=torch.float32, device="cuda:0"))
    assert ctx.launch_count() == before
    g = to_dev(gen.lego_scene(n=4).gaussians)
    for field, value in [(16, 0.0), (17, -1.0), (12, np.nan), (3, np.inf)]:
        bad = cam.copy()
        bad[field] = value
        with pytest.raises(gsr.GsrError) as ex:
            gsr.project_forward(ctx, g, bad)
        assert ex.value.code == 1


def test_projection_chain_matches_oracle_chain(gsr, ctx):
    """Projection, binning, forward, backward and projection backward on the
    GPU, against the oracle's projection backward of the oracle rasterizer's
    gradient, both fed the GPU-projected splats (the rasterizer's own parity
    tests fix that stage on identical inputs)."""
    sc = gen.lego_scene(n=20_000, seed=9)
    g = to_dev(sc.gaussians)
    sp, d = gsr.project_forward(ctx, g, sc.camera)
    wl = gen.from_arrays("chain", sc.width, sc.height, sp.cpu().numpy(), d.cpu().numpy(), seed=9)
    res = run_gpu(gsr, ctx, wl, backward=True)
    G_gpu = res["grad"]
    dg = gsr.project_backward(ctx, g, sc.camera, to_dev(G_gpu)).cpu().numpy()
    o = run_oracle(wl, backward=True)
    G_ref = o["bwd"]["grad"]
    # the rasterizer gradient's own tolerance, carried through the projection
    G_tol = GRAD_ATOL + GRAD_RTOL * np.abs(G_ref) + GRAD_COND * o["bwd"]["gabs"]
    knife = o["bwd"]["knife"]
    keep = ~knife
    proj_checks.check_backward(sc.gaussians[keep], sc.camera, G_ref[keep].astype(np.float32), dg[keep],
                               extra_G=G_tol[keep])


@pytest.mark.parametrize("seed", range(12))
def test_projection_random_cameras(gsr, ctx, seed):
    sc = gen.random_scene(seed)
    sp, d, grad = _project(gsr, ctx, sc.gaussians, sc.camera, sc.dl_dsplat)
    proj_checks.check_forward(sc.gaussians, sc.camera, sp, d)
    proj_checks.check_backward(sc.gaussians, sc.camera, sc.dl_dsplat, grad)
