"""The multi-rank path of bench.py on the CPU (gloo, world size 2): each rank
runs its own independent batch and only the timing is combined -- the
reported time is the max over ranks, the throughput counts every rank's work."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        elapsed = 1.0 + rank                      # rank 1 is slower
        worst = bench.max_over_ranks(elapsed, w)
        work = {"step_bytes": 100e9, "flops": 1e12, "tokens": 10}
        value, unit = bench.metric_value("decode", work, worst, w)
        q.put((r, w, local, worst, value, unit))
    finally:
        dist.destroy_process_group()


def test_timing_is_max_over_ranks_and_work_is_summed():
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
    for rank, (r, w, local, worst, value, unit) in enumerate(results):
        assert (r, w, local) == (rank, 2, rank)
        assert worst == 2.0                       # max over ranks
        assert unit == "GB/s"
        assert abs(value - 2 * 100.0 / 2.0) < 1e-9   # both ranks' bytes / slowest time


def test_reference_arm_runs_on_rank_0_only():
    """Under a multi-rank launch the oracle arm runs on rank 0 alone: another
    rank exits 0 at once, printing nothing and doing no work."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "3"],
                         cwd=root, env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""
