"""The multi-rank timing path of bench.py on CPU: two gloo ranks, each with
its own timed milliseconds; every rank must see the slowest rank's time, and
the whole-job throughput counts both ranks' bytes (weak scaling)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx = bench.reduce_max_ms(torch, 10.0 + 5.0 * rank, dist, torch.device("cpu"))
    val = bench.throughput(world, bench.STEP_BYTES, 100, mx)
    dist.barrier()
    queue.put((rank, mx, val))
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    for rank, mx, val in results:
        assert mx == 15.0
        assert val == pytest.approx(2 * bench.STEP_BYTES * 100 / 15e-3 / 1e9)
