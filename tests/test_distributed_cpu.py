"""The multi-rank path of bench.py on CPU (gloo, world size 2): every rank
joins the process group, the barrier completes, and the step time reported is
the maximum over ranks.  The FP4 path itself shards by tokens with no
data-path collective, so the ranks run independent replicas."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), FP4_BENCH_BACKEND="gloo")
    import bench
    r, local, w, pg = bench.dist_setup(world)
    assert (r, w) == (rank, world) and pg is not None
    bench.barrier(pg)
    t = bench.max_over_ranks(pg, 1.0 + 10.0 * rank)
    q.put((rank, t))
    pg.destroy_process_group()


def test_bench_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]
