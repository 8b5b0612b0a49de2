"""Replicas on several GPUs: the benchmark's host-side aggregation (barrier, the
maximum time over ranks, whole-job throughput) with two gloo ranks on the CPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        # rank r took (r + 1) ms for the device-timed step and (10 - r) ms end to end
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 300
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res[0] == res[1] == [2.0, 10.0]


def test_one_process_is_its_own_maximum():
    import bench
    assert bench.max_over_ranks([3.5, 1.25], "cpu") == [3.5, 1.25]


@pytest.mark.parametrize("n_gpus", [1, 2, 8])
def test_job_value_counts_every_rank_over_the_slowest(n_gpus):
    import bench
    # 48 layer-tokens per step, 400 steps per rank, the slowest rank 500 ms
    assert bench.job_value(n_gpus, 48 * 400, 500.0) == pytest.approx(n_gpus * 48 * 400 / 0.5)
