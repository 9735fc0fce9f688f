"""Race canary: a build of the library in which warps sleep pseudo-random
times at the staging barriers and candidate windows of the raster kernels and
the radix downsweep (GSR_RACE_CANARY) must give the same bits as the normal
build: binning, forward and the deterministic backward.  A shared-memory
access that relied on an interleaving no barrier enforces would show here."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def gsr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gaussian_splatting_tile_bin_gb300 as g
    return g


def test_race_canary_changes_no_bit(gsr, tmp_path):
    from gaussian_splatting_tile_bin_gb300 import build as b
    lib = b.build(out=str(tmp_path / "canary" / "libgsr.so"), extra_flags=["-DGSR_RACE_CANARY"])
    out = tmp_path / "canary.npz"
    env = dict(os.environ, GSR_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "race_canary_run.py"), str(out)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    sys.path.insert(0, HERE)
    import race_canary_run
    ref = race_canary_run.outputs()
    got = np.load(out)
    assert set(got.files) == set(ref)
    for k, v in ref.items():
        assert np.array_equal(got[k].view(np.uint8), np.ascontiguousarray(v).view(np.uint8)), k
