"""The N > 1 bench path on CPU: two gloo ranks, one process each (spawned),
as torchrun would start them.  Every rank runs its own replica of the step
(the attention of each (batch, head) is independent, so nothing is
exchanged); the job's step time is the slowest rank's, and its throughput
counts the work of every rank.  The reference arm does its work on rank 0
only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD))
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        ms = [2.5, 4.0][rank]  # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, dist, "cpu")
        value = bench.whole_job_tflops(WORLD, 1e12, ms_max)
        ref = bench.run_reference(argparse.Namespace(workload="bert_large", steps=1, warmup=3),
                                  rank, WORLD) if rank != 0 else "skipped"
        dist.barrier()
        out.put((rank, ms_max, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_every_replica():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, out)) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(out.get() for _ in range(WORLD))
    for rank, ms_max, value, ref in got:
        assert ms_max == 4.0, (rank, ms_max)
        # 2 ranks x 1 TFLOP each in 4 ms
        assert value == pytest.approx(WORLD * 1e12 / 4e-3 / 1e12)
    assert got[1][3] is None  # the reference arm: no work off rank 0


def test_one_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.whole_job_tflops(1, 2e12, 2.0) == pytest.approx(1000.0)
