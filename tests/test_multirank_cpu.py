"""The bench's N > 1 path on CPU: two gloo ranks (one process each, 127.0.0.1) run the
bench's own barrier and max-over-ranks, and the whole-job rate of independent replicas is
every rank's units over the slowest rank's time.  No GPU is needed."""
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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each rank's timed region; the slowest one defines the job's time
        seconds = [0.50, 0.75][rank]
        slowest = bench.max_over_ranks(world, seconds, device="cpu")
        out[rank] = (slowest, bench.whole_job_rate(100.0, world, slowest))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_rate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        res = dict(out)
    # both ranks agree on the slowest rank's time and on the whole-job rate
    assert res[0] == res[1] == (0.75, pytest.approx(100.0 * 2 / 0.75))


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1, 1.25) == 1.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
