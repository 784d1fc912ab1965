"""The core pin, on the GPU: rounds run through libdspark.so emit tokens that follow the
target law (numb3r33 blog "One-token exactness", "Speculative sampling in one picture":
the law of every emitted token is the target's softmax, whatever the draft law and the
verify lengths).

(1) V=8, gamma=3, batches of R=2 requests, 10^6 trials: the draft and verification of
    every trial run on the device (many trials per call: a request's draws depend only
    on its own request id, never on the batch layout), and the scheduler runs on the
    device once per 2-request batch (a CUDA graph of 1000 scheduler calls, replayed over
    the batches).  The emitted y_m, given that the round emitted at least m tokens,
    follow softmax(target row m-1 / T) (chi-square, p > 1e-5), for the early-stop and
    capacity-K schedulers and a non-unit temperature.
(2) A bf16 tensor-core shape (V=1024, rank 64): the first-position acceptance rate over
    10^6 trials equals sum_v min(p, q) = 1 - TV(p, q) computed in fp64 from the same bf16
    inputs, within 5 sigma.
"""
import math

import numpy as np
import pytest
import torch
from scipy import special

from tests.test_oracle_law import GAMMA, D, V, _check_law, _problem

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N = 1_000_000
CHUNK = 65536  # requests per draft / verify call (CUDA-core path: R*gamma <= 262140)
GRAPH_CALLS = 1000  # scheduler calls per captured graph


def _b():
    from speculative_decoding_draft_03_gb300 import binding
    return binding


def _draft_and_verify_chunks(P, T, n, seed, rnd, ell_fn):
    """Draft every trial in chunks; ell_fn(conf [chunk, gamma] on the device, lo) returns the
    verify lengths for those trials; verification runs on the same chunks."""
    b = _b()
    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    U1, h1, tg1 = t(P["U"]), t(P["h"]), t(P["target"])
    W1, W2, cw = t(P["W1"]), t(P["W2"]), t(P["cw"])
    ctemp = torch.ones(GAMMA, device=dev)
    out = dict(x=[], n_acc=[], tokens=[], n_out=[], ell=[])
    for lo in range(0, n, CHUNK):
        m = min(CHUNK, n - lo)
        U = U1.expand(m, GAMMA, V).contiguous()
        h = h1.expand(m, GAMMA, D).contiguous()
        target = tg1.expand(m, GAMMA + 1, V).contiguous()
        ids = torch.arange(lo, lo + m, dtype=torch.int64, device=dev)
        x0 = torch.full((m,), P["x0"], dtype=torch.int32, device=dev)
        d = b.markov_draft(U, W1, W2, h, cw, 0.0, 1.0, ctemp, T, x0, ids, seed, rnd)
        ell = ell_fn(d["conf"], lo)
        v = b.verify(target, U, W1, W2, x0, d["x"], d["logq"], d["lse"], ell, T, ids, seed, rnd)
        torch.cuda.synchronize()
        out["x"].append(d["x"].cpu().numpy())
        out["ell"].append(ell.cpu().numpy())
        for k in ("n_acc", "tokens", "n_out"):
            out[k].append(v[k].cpu().numpy())
    return {k: np.concatenate(a, 0) for k, a in out.items()}


class _BatchScheduler:
    """dspark_schedule on consecutive 2-request batches: GRAPH_CALLS calls captured once on
    a staging buffer, replayed for every group of batches."""

    def __init__(self, R, sps, mode, with_hist):
        b = _b()
        dev = torch.device("cuda")
        self.R = R
        self.conf = torch.zeros((GRAPH_CALLS, R, GAMMA), dtype=torch.float32, device=dev)
        self.hist = torch.zeros_like(self.conf) if with_hist else None
        self.ell = torch.zeros((GRAPH_CALLS, R), dtype=torch.int32, device=dev)
        self.B = torch.zeros((GRAPH_CALLS, 1), dtype=torch.int32, device=dev)
        self.tau = torch.zeros((GRAPH_CALLS, 1), dtype=torch.float64, device=dev)
        self.sps = torch.from_numpy(sps).to(dev)
        self.ws = b.workspace(b.schedule_workspace_size(R, GAMMA), dev)

        def calls():
            for i in range(GRAPH_CALLS):
                b.schedule(self.conf[i], self.sps, mode, None if self.hist is None else self.hist[i], 0,
                           out=dict(ell=self.ell[i], B=self.B[i], tau=self.tau[i]), ws=self.ws)

        calls()  # eager once (also validates the arguments)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(self.graph, stream=side):
            calls()
        torch.cuda.current_stream().wait_stream(side)

    def __call__(self, conf, hist):
        """conf [n, gamma] (n a multiple of R * GRAPH_CALLS) -> ell [n]."""
        n = conf.shape[0]
        per = self.R * GRAPH_CALLS
        assert n % per == 0
        out = torch.empty(n, dtype=torch.int32, device=conf.device)
        for lo in range(0, n, per):
            self.conf.copy_(conf[lo:lo + per].view(GRAPH_CALLS, self.R, GAMMA))
            if self.hist is not None:
                self.hist.copy_(hist[lo:lo + per].view(GRAPH_CALLS, self.R, GAMMA))
            self.graph.replay()
            out[lo:lo + per].copy_(self.ell.view(-1))
        return out


@pytest.mark.parametrize("mode,T", [(0, 1.0), (2, 1.0), (0, 0.7)])
def test_gpu_rounds_emit_target_law_1e6_trials(mode, T):
    b = _b()
    P = _problem(1, T)
    R = 2
    sps = 100.0 / (1.0 + np.arange(R * (GAMMA + 1) + 1) / 50.0)
    hist = None
    if mode == b.CAPACITY_K:
        rng = np.random.default_rng(9)
        hist = torch.from_numpy(rng.uniform(0.2, 1.0, (N, GAMMA)).astype(np.float32)).cuda()
    sched = _BatchScheduler(R, sps, mode, hist is not None)
    # the draft of every trial first (the scheduler needs whole groups of batches); this
    # first pass verifies with zero lengths, its results are not used
    dev = torch.device("cuda")
    confs = []

    def keep_conf(conf, lo):
        confs.append(conf.clone())
        return torch.zeros(conf.shape[0], dtype=torch.int32, device=dev)

    n = (N // (R * GRAPH_CALLS)) * R * GRAPH_CALLS
    _draft_and_verify_chunks(P, T, n, 3, 5, keep_conf)
    conf = torch.cat(confs, 0)
    ell = sched(conf, hist)
    ell_h = ell.cpu().numpy()
    assert (ell_h >= 0).all() and (ell_h <= GAMMA).all()
    assert len(np.unique(ell_h)) > 1  # the scheduler actually varies the length
    # the same drafts (same ids, seed and round) verified with the scheduled lengths
    out = _draft_and_verify_chunks(P, T, n, 3, 5, lambda c, lo: ell[lo:lo + c.shape[0]].contiguous())
    assert np.array_equal(out["ell"], ell_h)
    p_t = [special.softmax(P["target"][m].astype(np.float64) / T) for m in range(GAMMA + 1)]
    _check_law(out, p_t, n)
    n_acc = out["n_acc"]
    assert (out["n_out"] == n_acc + 1).all()
    assert (n_acc <= ell_h).all()
    for j in range(GAMMA):
        sel = n_acc > j
        assert (out["tokens"][sel, j] == out["x"][sel, j]).all()


def _bf16_bits(a):
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t, t.view(torch.int16).numpy().view(np.uint16)


def test_tensor_core_first_position_acceptance_rate():
    """bf16 factors on the tensor-core path: P(accept position 1) = sum_v min(p_v, q_v)."""
    b = _b()
    Vt, rank, dd = 1024, 64, 16
    rng = np.random.default_rng(11)
    Ut = rng.normal(0, 1.5, (1, Vt)).astype(np.float32)
    tgt = np.concatenate([Ut, Ut], 0) + rng.normal(0, 0.8, (2, Vt)).astype(np.float32)
    W1t, W1bits = _bf16_bits(rng.normal(0, 0.15, (Vt, rank)))
    W2t, W2bits = _bf16_bits(rng.normal(0, 0.15, (rank, Vt)))
    x0v = 17
    # fp64 laws from the exact bf16 inputs
    f = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q = special.softmax(Ut[0].astype(np.float64) + f(W1bits)[x0v] @ f(W2bits))
    p = special.softmax(tgt[0].astype(np.float64))
    alpha = np.minimum(p, q).sum()
    assert abs(alpha - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
    dev = torch.device("cuda")
    m = 131072
    U = torch.from_numpy(Ut).to(dev).view(1, 1, Vt).expand(m, 1, Vt).contiguous()
    target = torch.from_numpy(tgt).to(dev).view(1, 2, Vt).expand(m, 2, Vt).contiguous()
    W1, W2 = W1t.to(dev), W2t.to(dev)
    h = torch.zeros((m, 1, dd), dtype=torch.bfloat16, device=dev)
    cw = torch.zeros(dd + rank, device=dev)
    ctemp = torch.ones(1, device=dev)
    x0 = torch.full((m,), x0v, dtype=torch.int32, device=dev)
    ell = torch.ones(m, dtype=torch.int32, device=dev)
    accepted, n = 0, 0
    for lo in range(0, N, m):
        ids = torch.arange(lo, lo + m, dtype=torch.int64, device=dev)
        d = b.markov_draft(U, W1, W2, h, cw, 0.0, 1.0, ctemp, 1.0, x0, ids, 21, 4)
        v = b.verify(target, U, W1, W2, x0, d["x"], d["logq"], d["lse"], ell, 1.0, ids, 21, 4)
        accepted += int((v["n_acc"] >= 1).sum())
        n += m
    torch.cuda.synchronize()
    rate = accepted / n
    assert abs(rate - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / n), (rate, alpha)
