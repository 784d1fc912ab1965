"""The full-size workloads, in the launch configuration the benchmark times (one CUDA graph
per round), checked against the fp64 oracle on every request.

The oracle recomputes every request's draft at the full vocabulary and hidden sizes; where
a draw is a boundary case (the oracle's key margin below 1e-5, the GPU holding the runner-
up) the oracle adopts the GPU's token and recomputes that request's later positions from
it, so every draw is compared.  The scheduler runs on the GPU's own confidences (its
exact fp32 inputs) for the whole batch, and verification on the GPU's drafts and verify
lengths for every request.  The stress workload also runs chained rounds: x0 of round
t+1 is the last token the GPU emitted in round t (the RNG round index advances).
"""
import numpy as np
import pytest
import torch

from speculative_decoding_draft_03_gb300 import workloads as wl
from tests.parity import Tally, check_round_stagewise

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROUND = 17


def _host(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _gpu_round(rd, rnd, x0=None):
    g = rd.capture(rnd=rnd, x0=x0)
    g.replay()
    torch.cuda.synchronize()
    assert rd.status() == 0
    d = {k: v.cpu().numpy() for k, v in rd.draft_out.items()}
    s = {k: v.cpu().numpy() for k, v in rd.sched_out.items()}
    v = {k: t.cpu().numpy() for k, t in rd.verify_out.items()}
    return d, s, v


@pytest.mark.parametrize("name", ["qwen3-8b", "batch128", "deepseek-v4"])
def test_full_size_round_on_every_request(name):
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make(name, device="cuda")
    rd = b.Round(w)
    d, s, v = _gpu_round(rd, ROUND)
    wn = wl.to_numpy(w)
    tally = Tally()
    check_round_stagewise(w, wn, d, s, v, ROUND, wn["x0"], tally)
    tally.check_rate()
    assert tally.draws >= w["R"] * w["gamma"]


def test_full_size_stress_chained_rounds():
    """Five chained full-size stress rounds (R=512, gamma=15, V=151936), every request."""
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make("stress", device="cuda")
    rd = b.Round(w)
    wn = wl.to_numpy(w)
    x0 = w["x0"].clone()
    tally = Tally()
    R = w["R"]
    for t in range(5):
        x0_h = x0.cpu().numpy()
        d, s, v = _gpu_round(rd, t, x0=x0)
        check_round_stagewise(w, wn, d, s, v, t, x0_h, tally)
        last = v["tokens"][np.arange(R), v["n_out"] - 1]
        x0 = torch.from_numpy(last.astype(np.int32)).cuda()
    tally.check_rate()
    assert tally.draws >= 5 * R * w["gamma"]
