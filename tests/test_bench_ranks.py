"""Multi-process host logic of bench.py on CPU: with `gloo` and world size 2,
every rank joins the barrier, the step time is the maximum over ranks and the
token count the sum (the whole-job aggregate the bench line reports)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CF_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    r, w, local, pg = bench.dist_setup(world)
    bench.barrier(pg)
    ms = bench.max_over_ranks(pg, 10.0 + 5.0 * r)      # rank r took 10 + 5r ms
    tok = bench.sum_over_ranks(pg, 1000.0 * (r + 1))    # and processed 1000 (r + 1) tokens
    bench.barrier(pg)
    q.put((r, w, local, ms, tok))
    pg.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_bench_aggregates_over_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(world))
    for r, (rank, w, local, ms, tok) in enumerate(got):
        assert (rank, w, local) == (r, world, r)
        assert ms == 10.0 + 5.0 * (world - 1)             # the slowest rank's time
        assert tok == 1000.0 * world * (world + 1) / 2    # all ranks' tokens


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    rank, world, local, pg = bench.dist_setup(1)
    assert (rank, world, local, pg) == (0, 1, 0, None)
    assert bench.max_over_ranks(None, 3.5) == 3.5 and bench.sum_over_ranks(None, 7.0) == 7.0
