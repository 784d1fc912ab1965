"""The full-size workloads, in the launch configuration the benchmark times (one CUDA graph
per round), checked against the fp64 oracle on sampled requests.

Requests are independent in the draft and verify stages, so the oracle recomputes a few
sampled requests at the full vocabulary and hidden sizes: their draft outputs, and their
verification given the GPU's drafts and verify lengths.  The scheduler is global; its
inputs are only the R x gamma confidences, so the oracle runs it on the GPU's own
confidences for the whole batch.  Inputs are generated on the device (the same seeded
recipes); the oracle gets host copies of the sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_03_gb300 import workloads as wl
from tests.parity import Tally, compare_draft, compare_schedule, compare_verify

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROUND = 17


def _host(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@pytest.mark.parametrize("name", ["qwen3-8b", "batch128", "deepseek-v4", "stress"])
def test_full_size_round_on_sampled_requests(name):
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make(name, device="cuda")
    R, gamma = w["R"], w["gamma"]
    rd = b.Round(w)
    g = rd.capture(rnd=ROUND)
    g.replay()
    torch.cuda.synchronize()
    assert rd.status() == 0
    d = {k: v.cpu().numpy() for k, v in rd.draft_out.items()}
    s = {k: v.cpu().numpy() for k, v in rd.sched_out.items()}
    v = {k: t.cpu().numpy() for k, t in rd.verify_out.items()}
    bf = any(w[k].dtype == torch.bfloat16 for k in ("U", "target", "W1", "W2"))
    tol = 2e-3 if bf else 1e-5
    tally = Tally()

    # sampled requests: first, middle, last
    rows = np.array(sorted({0, R // 2, R - 1}))
    idx = torch.from_numpy(rows).cuda()
    sub = {k: _host(w[k].index_select(0, idx)) for k in ("U", "target", "h", "x0", "req_id")}
    W1, W2 = _host(w["W1"]), _host(w["W2"])
    conf_w, conf_temp = _host(w["conf_w"]), _host(w["conf_temp"])

    ref_d = oracle.markov_draft(sub["U"], W1, W2, sub["h"], conf_w, w["conf_b"], w["conf_logit_scale"], conf_temp,
                                w["temperature"], sub["x0"], sub["req_id"], w["seed"], ROUND)
    compare_draft({k: d[k] for k in ("x", "logq", "lse", "conf")}, ref_d, tol, tally, rows=rows)

    # the scheduler on the GPU's confidences (its exact fp32 inputs)
    hist = None if w["conf_hist"] is None else _host(w["conf_hist"])
    ref_s = oracle.schedule(d["conf"], _host(w["sps"]), w["mode"], hist, w.get("fixed_len", 0))
    compare_schedule(dict(ell=s["ell"], B=s["B"][0], tau=s["tau"][0]), ref_s, tally, tau_tol=1e-9)

    # verification of the sampled requests given the GPU's drafts and verify lengths
    ref_v = oracle.verify(sub["target"], sub["U"], W1, W2, sub["x0"], d["x"][rows], d["logq"][rows],
                          d["lse"][rows], s["ell"][rows], w["temperature"], sub["req_id"], w["seed"], ROUND)
    compare_verify(v, ref_v, tally, rows=rows)
    tally.check_rate()
    # every request's output is well formed
    assert ((v["n_acc"] >= 0) & (v["n_acc"] <= s["ell"])).all()
    assert (v["n_out"] == v["n_acc"] + 1).all()
    assert int(s["B"][0]) == R + int(s["ell"].sum())
