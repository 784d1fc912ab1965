"""The recurrent draft head (dspark_rnn_draft / dspark_verify_rnn) against the fp64 oracle.

Each position is checked given the GPU's own previous state and token (the chain is a
sequence of decisions; conditioning on the GPU's path keeps one boundary decision from
spreading):
* the stored state s_k equals the oracle's cell output rounded to the storage type: for
  bf16 up to one unit in the last place where the fp32 cell sits on a rounding boundary
  (counted, rare; within 1e-6 near zero); for fp32 storage within 1e-6 (the fp32 cell's
  own rounding);
* the draw given the GPU's s_k is the oracle's draw (bit-exact, boundary cases counted),
  with lse / logq / c_k within the probability tolerances;
* verification given the GPU's drafts and states is the oracle's, token for token.
Shapes cover the CUDA-core path (fp32), the tensor-core path with one and several
request blocks, bf16 logits, a hidden width with two projection splits and a ragged one,
and the full Qwen3-8B-shaped workload on sampled requests.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_03_gb300 import workloads as wl
from tests.parity import BOUNDARY, Tally, close, compare_verify

pytestmark = pytest.mark.gpu


def _host(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _ulp(v, bf16):
    """One unit in the last place of the storage type at |v| (bf16: 8 significant bits)."""
    m = 8 if bf16 else 24
    e = np.floor(np.log2(np.maximum(np.abs(v), 1e-30)))
    return np.exp2(e - (m - 1))


def _check_positions(w, d, rnd, rows, tally, tol):
    """Per-position comparison of requests `rows` given the GPU's path."""
    bf16 = w["Wo"].dtype == torch.bfloat16
    Hn = {k: _host(w[k]) for k in ("E", "Wse", "Wh", "Wo", "bgc", "conf_w", "conf_temp")}
    state = _host(d["state"])
    sg = _f64(state)
    x = _host(d["x"])
    lse, logq, conf = _host(d["lse"]), _host(d["logq"]), _host(d["conf"])
    x0 = _host(w["x0"])
    gamma, ns = w["gamma"], w["ns"]
    n_el = n_ulp = 0
    idx = torch.as_tensor(rows, device=w["U"].device)
    U = _host(w["U"].index_select(0, idx))
    h = _host(w["h"].index_select(0, idx))
    req = _host(w["req_id"])
    cref = oracle.rnn_confidence(h, sg[rows], Hn["conf_w"], w["conf_b"], w["conf_logit_scale"], Hn["conf_temp"])
    for i, r in enumerate(rows):
        for k in range(1, gamma + 1):
            s_prev = np.zeros(ns) if k == 1 else sg[r, k - 2]
            x_prev = x0[r] if k == 1 else x[r, k - 2]
            s_ref = oracle.rnn_cell(s_prev, x_prev, Hn["E"], Hn["Wse"], Hn["Wh"], Hn["bgc"], h[i, k - 1])
            diff = np.abs(sg[r, k - 1] - s_ref)
            n_el += ns
            if bf16:
                # fp32 cell, one rounding to bf16: equal, or one unit apart at a rounding boundary
                # (near zero, where a bf16 unit is below the fp32 cell's own error, within 1e-6)
                n_ulp += int((diff > 0).sum())
                assert (diff <= np.maximum(1.01 * _ulp(s_ref, True), 1e-6)).all(), (r, k, diff.max())
            else:
                # fp32 state: the fp32 cell's own error (a few 1e-8 on values below 1)
                assert (diff <= 1e-6).all(), (r, k, diff.max())
            ref = oracle.draft_row(U[i, k - 1], sg[r, k - 1], Hn["Wo"], w["temperature"], w["seed"], req[r], rnd, k)
            tally.draws += 1
            if x[r, k - 1] != ref["x"]:
                assert ref["margin"] < BOUNDARY and x[r, k - 1] == ref["runner_up"], (r, k, ref)
                tally.boundary += 1
            else:
                assert not close(logq[r, k - 1], ref["logq"], tol, 1.0), (r, k, logq[r, k - 1], ref["logq"])
            assert not close(lse[r, k - 1], ref["lse"], tol, 1.0), (r, k, lse[r, k - 1], ref["lse"])
            assert not close(conf[r, k - 1], cref[i, k - 1], tol, 1e-12), (r, k, conf[r, k - 1], cref[i, k - 1])
    # states one unit off (an fp32 cell output next to a rounding boundary) stay rare
    assert n_ulp <= max(4, 2e-3 * n_el), (n_ulp, n_el)


def _rnn_workload(name, **over):
    return wl.add_rnn_head(wl.make(name, device="cuda", **over))


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),                                            # CUDA cores, fp32
    ("qwen3-8b", dict(R=5, gamma=4, V=2056, d=64)),          # tensor cores, ragged vocabulary tail
    ("deepseek-v4", dict(R=40, gamma=3, V=1288, d=600)),     # bf16 logits, 64-request block, 2 splits
    ("stress", dict(R=140, gamma=3, V=1032, d=64)),          # two 128-request blocks
])
def test_rnn_round_matches_oracle(name, over):
    from speculative_decoding_draft_03_gb300 import binding as b
    w = _rnn_workload(name, **over)
    rd = b.Round(w)
    rnd = 4
    d, s, v = rd.run(rnd=rnd)
    torch.cuda.synchronize()
    assert rd.status() == 0
    bf = any(w[k].dtype == torch.bfloat16 for k in ("U", "target", "Wo"))
    tol = 2e-3 if bf else 1e-5
    tally = Tally()
    R = w["R"]
    rows = np.arange(R) if R <= 40 else np.array(sorted({0, 1, 63, 64, 127, 128, R - 1}))
    _check_positions(w, d, rnd, rows, tally, tol)
    # verification given the GPU's drafts, verify lengths and states
    idx = torch.as_tensor(rows, device="cuda")
    sub = {k: _host(w[k].index_select(0, idx)) for k in ("U", "target", "x0", "req_id")}
    dn = {k: _host(t) for k, t in d.items()}
    ell = _host(s["ell"])
    ref_v = oracle.verify(sub["target"], sub["U"], np.zeros((1, 1), np.float32), _host(w["Wo"]), sub["x0"],
                          dn["x"][rows], dn["logq"][rows], dn["lse"][rows], ell[rows], w["temperature"],
                          sub["req_id"], w["seed"], rnd, state=_f64(dn["state"][rows]))
    compare_verify({k: _host(t) for k, t in v.items()}, ref_v, tally, rows=rows)
    tally.check_rate()


def test_rnn_graph_replay_equals_eager():
    from speculative_decoding_draft_03_gb300 import binding as b
    w = _rnn_workload("qwen3-8b", R=20, gamma=5, V=4104, d=128)
    rd = b.Round(w)
    d, s, v = rd.run(rnd=9)
    torch.cuda.synchronize()
    ref = {k: t.clone() for k, t in list(d.items()) + list(v.items())}
    g = rd.capture(rnd=9)
    g.replay()
    torch.cuda.synchronize()
    for k, t in list(rd.draft_out.items()) + list(rd.verify_out.items()):
        assert torch.equal(t, ref[k]), k


@pytest.mark.slow
def test_rnn_full_size_sampled_requests():
    from speculative_decoding_draft_03_gb300 import binding as b
    w = _rnn_workload("qwen3-8b")
    rd = b.Round(w)
    d, s, v = rd.run(rnd=2)
    torch.cuda.synchronize()
    assert rd.status() == 0
    tally = Tally()
    R = w["R"]
    _check_positions(w, d, 2, np.array([0, R // 2, R - 1]), tally, 2e-3)
    tally.check_rate()


@pytest.mark.parametrize("name,over", [("tiny", {}), ("qwen3-8b", dict(R=6, gamma=3, V=2056, d=64))])
def test_rnn_without_hidden_state_or_embedding(name, over):
    # d = 0 (no hidden-state path, no projection) and ne = 0 (no embedding): the cell runs
    # on the state alone; each position checked given the GPU's previous state
    from speculative_decoding_draft_03_gb300 import binding as b
    w = _rnn_workload(name, **over)
    R, gamma, ns = w["R"], w["gamma"], w["ns"]
    dev = w["U"].device
    Wse = w["Wse"][:ns].contiguous()  # state rows only
    h0 = torch.zeros((R, gamma, 0), dtype=w["h"].dtype, device=dev)
    Wh0 = torch.zeros((0, 2 * ns), dtype=w["Wse"].dtype, device=dev)
    conf_w = w["conf_w"][w["d"]:].contiguous()  # the state part only
    x0 = w["x0"]
    out = b.rnn_draft(w["U"], None, Wse, Wh0, w["bgc"], w["Wo"], h0, conf_w, w["conf_b"], w["conf_logit_scale"],
                      w["conf_temp"], w["temperature"], x0, w["req_id"], w["seed"], 7)
    torch.cuda.synchronize()
    bf16 = w["Wo"].dtype == torch.bfloat16
    sg = _f64(_host(out["state"]))
    x = _host(out["x"])
    E0 = np.zeros((w["V"], 0), np.uint16 if bf16 else np.float32)
    hrow = np.zeros(0, np.uint16 if bf16 else np.float32)
    U = _host(w["U"])
    conf = oracle.rnn_confidence(np.zeros((R, gamma, 0), np.float32), sg, _host(conf_w), w["conf_b"],
                                 w["conf_logit_scale"], _host(w["conf_temp"]))
    tol = 2e-3 if bf16 else 1e-5
    boundary = 0
    for r in range(R):
        for k in range(1, gamma + 1):
            s_prev = np.zeros(ns) if k == 1 else sg[r, k - 2]
            s_ref = oracle.rnn_cell(s_prev, 0, E0, _host(Wse), _host(Wh0), _host(w["bgc"]), hrow)
            lim = np.maximum(1.01 * _ulp(s_ref, True), 1e-6) if bf16 else 1e-6
            assert (np.abs(sg[r, k - 1] - s_ref) <= lim).all(), (r, k)
            ref = oracle.draft_row(U[r, k - 1], sg[r, k - 1], _host(w["Wo"]), w["temperature"], w["seed"], r, 7, k)
            if x[r, k - 1] != ref["x"]:
                assert ref["margin"] < BOUNDARY and x[r, k - 1] == ref["runner_up"]
                boundary += 1
            assert abs(_host(out["conf"])[r, k - 1] - conf[r, k - 1]) <= tol * max(conf[r, k - 1], 1e-12)
    assert boundary <= 1
