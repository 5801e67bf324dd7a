"""bench.py's multi-rank logic on the CPU (gloo, world size 2).

With N GPUs the bench runs N independent replicas (the path needs no
exchange): every rank times its own steps, the timed region is the slowest
rank's, the value is every rank's units over that time, and only rank 0
prints.  The reference arm runs on rank 0 alone; the other ranks exit
without work.  Two spawned processes check these rules with the gloo
backend on 127.0.0.1.
"""
import io
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                          WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
        import torch
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo", rank=rank, world_size=world)
        slowest = bench.max_over_ranks(torch, 1.0 + rank, world, "cpu")  # rank r took 1 + r seconds
        rate = bench.whole_job_rate(100.0, 3, world, slowest)
        out = io.StringIO()
        if rank != 0:
            with redirect_stdout(out):
                r = bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "2"]))
            assert r is None
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, slowest, rate, out.getvalue()))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, None, repr(e)))


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in procs:
            rank, slowest, rate, text = q.get(timeout=120)
            results[rank] = (slowest, rate, text)
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    assert set(results) == {0, 1}, results
    for rank, (slowest, rate, text) in results.items():
        assert slowest == 2.0, (rank, text)          # the slower rank's time, on both ranks
        assert rate == 2 * 100.0 * 3 / 2.0           # both ranks' units over that time
    assert results[1][2] == ""                        # rank 1 of the reference arm: no work, no output
