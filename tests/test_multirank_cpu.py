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


def test_bench_launcher_starts_one_rank_per_gpu():
    """bench.py --gpus 2, run without torchrun, relaunches itself under
    torch.distributed.run with two ranks; with --launcher-check the ranks form
    a gloo group, reduce their times and rank 0 alone prints the whole-job
    figure."""
    import json
    import subprocess
    import sys
    import bench
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2", "--launcher-check"],
                       capture_output=True, text=True, timeout=240, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["world"] == 2 and lines[0]["max_ms"] == 15.0
    assert lines[0]["value"] == pytest.approx(2 * bench.STEP_BYTES / 15e-3 / 1e9)
