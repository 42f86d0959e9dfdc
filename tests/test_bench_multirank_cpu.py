"""The multi-rank side of bench.py on the CPU: two gloo ranks (the GPU run
uses one NCCL rank per GPU with the same calls).  Ranks run replicas with no
exchange on the data path; the timing takes the slowest rank, and the
whole-job figure divides its time by all ranks' steps."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        bench.barrier(world)
        # rank r spent 10 (r + 1) ms on 5 steps: the slowest rank sets the pace
        job_us, ms_per_step = bench.job_us_per_step(10.0 * (rank + 1), 5, world)
        bench.barrier(world)
        results[rank] = (job_us, ms_per_step, bench.reduce_max(float(rank), world))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_count_all_steps():
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        job_us, ms_per_step, top = results[r]
        assert ms_per_step == pytest.approx(4.0)   # max(10, 20) ms / 5 steps
        assert job_us == pytest.approx(2000.0)     # 4 ms per step over 2 ranks' steps
        assert top == 1.0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_us_per_step(40.0, 5, 1) == pytest.approx((8000.0, 8.0))
    bench.barrier(1)  # no-op without a process group
