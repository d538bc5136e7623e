"""Host-side N > 1 logic of the bench on CPU: world size 2 over gloo.

Every GPU runs an independent replica of the simulated job, so the only
cross-rank logic is the timing: the slowest rank's step time, and the whole-job
value = bytes of all replicas / that time.  The reference arm runs on rank 0
alone; other ranks exit without work."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 2.0 + rank * 3.5                      # rank 1 is slower
        m = bench.max_over_ranks(ms)
        v = bench.whole_job_gbs(10 ** 9, world, m)
        q.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.5, 5.5]              # both ranks see the slowest time
    assert res[0][2] == pytest.approx(2 * 1e9 / 5.5e-3 / 1e9)


def test_reference_arm_rank_nonzero_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=120, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_single_process_helpers_without_a_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_gbs(4 * 10 ** 9, 1, 2.0) == pytest.approx(2000.0)
