"""The N > 1 path of bench.py on CPU: world-size-2 gloo process group, max-over-ranks timing,
and the reference arm printing on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank]
        got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == [2.0, 10.0] and results[1] == [2.0, 10.0]


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], None, None) == [3.0, 4.0]


def test_reference_arm_other_ranks_are_silent(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload = "llama8b-int4a-decode"
        m = 0
        steps = 1
        warmup = 3
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, rank=1, world=2)
    assert buf.getvalue() == ""
