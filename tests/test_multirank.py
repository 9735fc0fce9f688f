"""bench.py's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.

With N GPUs the bench runs N independent replicas (the path has no exchange
step); the ranks only agree on the slowest rank's time.  These tests run that
agreement, and the reference arm's rank filter, in two real processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r ran 5 steps taking 10 (r + 1) ms in all.
        value = bench.job_ms_per_iter(10.0 * (rank + 1), 5, world)
        peak = bench.reduce_max(float(rank), world)
        # Only rank 0 runs the reference arm; the others return at once.
        ref_rc = bench.reference_arm(bench.parse_args(["--impl", "reference"])) if rank else None
        dist.barrier()
    finally:
        dist.destroy_process_group()
    results[rank] = (value, peak, ref_rc)


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        got = dict(results)
    # Slowest rank: 20 ms for 5 steps; the job made 2 x 5 iterations.
    assert got[0][0] == pytest.approx(2.0) and got[1][0] == pytest.approx(2.0)
    assert got[0][1] == 1.0 and got[1][1] == 1.0
    assert got[1][2] == 0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_ms_per_iter(12.0, 4, 1) == pytest.approx(3.0)
    assert bench.reduce_max(7.5, 1) == 7.5
