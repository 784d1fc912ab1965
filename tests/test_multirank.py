"""The N > 1 path of bench.py on CPU: two gloo ranks, each serving its own batch.  The
whole-job time is the slowest rank's, the tokens are summed, and the ranks' request ids
(hence their random streams) are disjoint.  The data path has no collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms, tok = bench.combine_ranks(10.0 + 5.0 * rank, 100 + rank, torch.device("cpu"))
        ids = bench.rank_request_ids(torch.arange(4, dtype=torch.int64), rank, 4)
        q.put((r, w, local, ms, tok, ids.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[:3] for x in res] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, ms, tok, _ in res:
        assert ms == 15.0 and tok == 201  # max time, summed tokens, on every rank
    assert set(res[0][5]).isdisjoint(res[1][5])
    assert res[0][5] == [0, 1, 2, 3] and res[1][5] == [4, 5, 6, 7]


def test_single_process_keeps_its_own_figures():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    assert bench.combine_ranks(3.5, 7, torch.device("cpu")) == (3.5, 7)
