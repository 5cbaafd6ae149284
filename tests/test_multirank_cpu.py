"""The N > 1 bench path on CPU: two gloo ranks on 127.0.0.1.

bench.py --gpus N runs one independent replica per rank (the layer does not
shard). The only cross-rank steps are the barrier around the timed region
and the max-over-ranks time; value is the bytes of all ranks over that time.
These tests run those steps with world_size 2 and the gloo backend.
"""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        t = bench.max_over_ranks(times[rank], world, "cpu")
        v = bench.whole_job_gbs(1_000_000_000, world, t)
        dist.barrier()
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def _run(times):
    world = len(times)
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


@pytest.mark.parametrize("times", [(3.0, 5.0), (7.5, 2.5)])
def test_max_over_ranks_and_whole_job_value(times):
    out = _run(list(times))
    slowest = max(times)
    for rank, t, v in out:
        assert t == slowest                              # every rank sees the slowest rank's time
        assert v == pytest.approx(2 * 1.0 / (slowest * 1e-3))   # 2 ranks x 1 GB over that time


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, 1, "cpu") == 4.0
    assert bench.whole_job_gbs(2_000_000_000, 1, 4.0) == pytest.approx(500.0)
