"""Helper of test_gpu_race_canary.py: runs binning, forward and the
deterministic backward on a few inputs with whichever libgsr.so GSR_LIBRARY
selects, and saves every output to the .npz named on the command line."""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import gen  # noqa: E402
import gaussian_splatting_tile_bin_gb300 as gsr  # noqa: E402
from gpu_helpers import run_gpu  # noqa: E402

WORKLOADS = {"small": gen.small, "lego_early": gen.lego_early, "elongated": gen.elongated_fixture}


def outputs():
    ctx = gsr.Context(0)
    ctx.set_option("deterministic", True)
    res = {}
    try:
        for name, make in WORKLOADS.items():
            g = run_gpu(gsr, ctx, make())
            for k in ("keys", "idx", "ranges", "out", "final_T", "last", "grad"):
                res[f"{name}.{k}"] = g[k]
    finally:
        ctx.close()
    torch.cuda.synchronize()
    return res


if __name__ == "__main__":
    np.savez(sys.argv[1], **outputs())
