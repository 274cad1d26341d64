"""The multi-process host path of bench.py on CPU (gloo, world size 2): the
slowest rank's time decides, and the whole-job rate counts every rank's work.
Also: the reference arm's non-zero ranks exit without work."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx = bench.dist_max(1.5 if rank == 0 else 4.0)
    rate = bench.whole_job_rate(1e12, mx, world)
    q.put((rank, mx, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, rate in res:
        assert mx == 4.0
        assert rate == pytest.approx(2 * 1e12 / 4e-3)


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.25) == 3.25
    assert bench.whole_job_rate(10.0, 2.0, 1) == pytest.approx(5000.0)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
