"""A batch split over the ranks of a process group with one global scheduler
(speculative_decoding_draft_03_gb300/sharded.py), host logic on CPU: two gloo ranks each
hold a slice of the batch's confidences, all-gather them, run the scheduler on the whole
batch and keep their slice of the verify lengths.  The concatenated slices, B and tau
equal the single-process scheduler on the whole batch (the oracle's scheduler stands in
for the library's on CPU; the GPU test of the same path uses the library)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(R, gamma, seed):
    rng = np.random.default_rng(seed)
    conf = rng.uniform(0.05, 0.99, (R, gamma)).astype(np.float32)
    conf[1, :] = 1.0  # exact ties across requests
    hist = rng.uniform(0.2, 1.0, (R, gamma)).astype(np.float32)
    sps = 1000.0 / (1.0 + np.arange(R * (gamma + 1) + 1) / 6.0)
    return conf, hist, sps


def test_partition_covers_the_batch():
    import sys
    sys.path.insert(0, ROOT)
    from speculative_decoding_draft_03_gb300.sharded import partition
    for R in (1, 2, 7, 512, 513):
        for world in (1, 2, 3, 8):
            parts = [partition(R, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == R
            for (a, b), (c, d) in zip(parts, parts[1:]):
                assert b == c and a <= b
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        partition(4, 2, 2)


def _worker(rank, world, port, q, R, gamma, mode):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from speculative_decoding_draft_03_gb300.sharded import gather_confidences, partition
        conf, hist, sps = _problem(R, gamma, 5)
        lo, hi = partition(R, world, rank)
        full = gather_confidences(torch.from_numpy(conf[lo:hi].copy()), R, world)
        same = bool(np.array_equal(full.numpy(), conf))
        s = oracle.schedule(full.numpy(), sps, mode, hist if mode == oracle.CAPACITY_K else None)
        q.put((rank, same, s["ell"][lo:hi].tolist(), s["B"], s["tau"]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("R,mode", [(7, 0), (12, 2), (9, 1)])
def test_two_gloo_ranks_schedule_like_one_process(R, mode):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    gamma = 5
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q, R, gamma, mode)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    conf, hist, sps = _problem(R, gamma, 5)
    ref = oracle.schedule(conf, sps, mode, hist if mode == oracle.CAPACITY_K else None)
    assert all(r[1] for r in res)  # every rank gathered the whole batch, in request order
    assert res[0][2] + res[1][2] == ref["ell"].tolist()
    for r in res:
        assert r[3] == ref["B"] and r[4] == ref["tau"]
    assert len(set(ref["ell"].tolist())) > 1
