"""The N > 1 bench path on CPU: two gloo ranks stand in for two GPUs.

Each rank runs the whole workload on its own device (replicas, weak scaling);
the only cross-rank step is the maximum of the timed quantities, after which
rank 0 reports units of all ranks divided by the slowest rank's time.  The
reference arm runs on rank 0 only.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (1 + r) s per step overall, 2 (r + 1) s compressing, 0.5 s retrieving
    t = bench.job_times([1.0 + rank, 2.0 * (rank + 1), 0.5], world, "cpu")
    v = bench.job_throughput(100.0, world, t[0])
    ref = bench.run_reference(None, rank, world) if rank != 0 else "rank0"
    q.put((rank, t, v, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_and_all_units():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {r: (t, v, ref) for r, t, v, ref in out}
    for r in (0, 1):
        t, v, _ = by_rank[r]
        assert t == [2.0, 4.0, 0.5]          # per-quantity maximum over the ranks
        assert v == pytest.approx(100.0)     # 2 ranks x 100 units / 2.0 s
    assert by_rank[1][2] is None             # the reference arm does no work off rank 0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_times([3.0, 1.0], 1, "cpu") == [3.0, 1.0]
    assert bench.job_throughput(50.0, 1, 2.0) == pytest.approx(25.0)
