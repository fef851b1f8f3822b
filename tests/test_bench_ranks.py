"""The bench's multi-rank arithmetic on CPU: two processes in a gloo group
(world_size 2, rendezvous on 127.0.0.1) take the largest per-rank time as the
job's time, and the job's GB/s counts the bytes of both replicas.  The GPU
bench runs the same functions over NCCL, one rank per GPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]          # rank 1 is the slow one
    m = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    v = bench.job_throughput(world, 1.0e9, m)
    out.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_bench_ranks_take_the_slowest_and_count_every_replica():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    out = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    for rank, m, v in got:
        assert m == 5.0                     # the job's time is the slowest rank's
        assert v == pytest.approx(400.0)    # 2 replicas x 1 GB per 5 ms


def test_bench_single_process_keeps_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, None, None) == 4.25
    assert bench.job_throughput(1, 447418368, 0.1042) == pytest.approx(447418368 / 0.1042e-3 / 1e9)


def test_reference_arm_runs_on_rank_0_only():
    """Under a multi-rank launch the reference arm's ranks other than 0 exit 0
    at once, printing nothing."""
    import subprocess
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
