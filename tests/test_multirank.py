"""The N > 1 path of bench.py on CPU: independent replicas, one rank per GPU, with the job's
time taken as the slowest rank's and the throughput summed over ranks (weak scaling).  The block
has no exchange step in its forward/backward pass, so no collective is in the data path; the
only cross-rank operations are the timing reduction and the barriers.  Run here as two gloo
ranks; the reference arm prints from rank 0 only."""

import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    my_ms = 10.0 * (rank + 1)                      # rank 1 is the slow one
    m = bench.max_over_ranks(my_ms)
    v = bench.job_throughput(5.0e12, world, m)
    dist.barrier()
    out.put((rank, m, v))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_sum_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 20.0                             # both ranks see the slowest time
        assert v == pytest.approx(2 * 5.0e12 / 0.020)  # units of both ranks / slowest time


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
