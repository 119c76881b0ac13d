"""The N > 1 path of bench.py on the CPU: two gloo ranks.

bench.py runs one replica per rank (the decode path shards by batch entry
with no exchange); what the ranks share is the timing: a barrier around the
timed region and the max over ranks of the elapsed time.  These tests run
that host logic with world_size 2 over gloo, without a GPU.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, values, out_q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        dist.barrier()
        got = bench.aggregate_max(values[rank], ws)
        # The reference arm prints on rank 0 only; the other ranks return at once.
        printed = ""
        if r != 0:
            buf = io.StringIO()
            with redirect_stdout(buf):
                bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1",
                                                      "--warmup", "0"]))
            printed = buf.getvalue()
        out_q.put((rank, ws, r, local, got, printed))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_over_ranks():
    world = 2
    values = [3.25, 7.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, values, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    for rank, ws, r, local, got, printed in results:
        assert ws == world and r == rank and local == rank
        assert got == max(values)
        if rank != 0:
            assert printed == ""


def test_single_rank_is_identity():
    assert bench.aggregate_max(1.5, 1) == 1.5
