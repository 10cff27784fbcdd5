"""The N>1 path of bench.py on CPU: two gloo ranks (127.0.0.1), each with its
own timing; the reported time is the slowest rank's and the throughput counts
every rank's tokens (weak scaling, replicas only).  The reference arm runs on
rank 0 alone; other ranks exit without work."""
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + 5.0 * rank, 3.0 - rank]          # rank 1 is slower in the first value
    got = bench.max_over_ranks(mine, "cpu")
    q.put((rank, got, bench.tokens_per_s(8192, 10, world, got[0])))
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_throughput_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tps in res:
        assert got == [15.0, 3.0]
        assert abs(tps - 8192 * 10 * 2 / 0.015) < 1e-6 * tps


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]
    assert bench.tokens_per_s(100, 2, 1, 1000.0) == 200.0


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
