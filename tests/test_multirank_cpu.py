"""The multi-rank path of bench.py on CPU: two gloo ranks, no GPU.

Every rank runs its own replica of the step (sequences are independent, so the path
shards with no data exchange); the only collective is the max over ranks of the
timed duration, from which rank 0 reports the whole-job rate.
"""
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed 10 steps in 100 * (r + 1) ms
        ms, rate = bench.job_rate(100.0 * (rank + 1), 10, world, "cpu")
        q.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, rate in got:
        assert abs(ms - 20.0) < 1e-9  # slowest rank: 200 ms / 10 steps
        assert abs(rate - world * 10 / 0.2) < 1e-9  # 20 layer-steps in 0.2 s


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
