"""The N > 1 benchmark path on CPU: two gloo ranks, independent replicas, the
job's throughput from the slowest rank, and the reference arm run by rank 0
only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.100, 0.125][rank]        # rank 1 is the slower replica
        value, ms = bench.replica_throughput(630_000_000, local_ms, world)
        q.put((rank, value, ms, bench.max_over_ranks(float(rank + 3), world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_from_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, ms, mx in out:
        assert ms == pytest.approx(0.125)
        assert value == pytest.approx(2 * 630_000_000 / 0.125e-3 / 1e9)
        assert mx == 4.0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
