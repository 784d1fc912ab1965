"""dspark_acceptance_overlap and dspark_verify_overlap against the fp64 oracle: c*_j =
sum_v min(q_j, p_j) for the drafted positions of a round, given the GPU's own drafted tokens
and draft normalisers (the fused call's verification also equals dspark_verify's).

Shapes cover both bias paths (tensor cores for bf16 factors, CUDA cores for fp32),
several vocabulary tiles with a ragged tail, more than one 128-row block of positions,
bf16 logits, lengths 0..gamma and no lengths at all; the full Qwen3-8B-shaped workload
is checked on sampled requests.  Tolerances are the ones stated for probabilities:
1e-5 relative with fp32 factors and logits, 2e-3 where any of them is bf16.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_03_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _host(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _check(got, ref, ell, tol):
    R, gamma = ref.shape
    for r in range(R):
        n = gamma if ell is None else int(ell[r])
        assert np.isnan(got[r, n:]).all() and np.isnan(ref[r, n:]).all()
        if n:
            err = np.abs(got[r, :n] - ref[r, :n])
            assert (err <= tol * np.maximum(1.0, np.abs(ref[r, :n]))).all(), (r, err.max())
            assert ((got[r, :n] >= -1e-6) & (got[r, :n] <= 1 + 1e-5)).all()


def _round(name, rnd, **over):
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make(name, device="cuda", **over)
    rd = b.Round(w)
    d, s, _ = rd.run(rnd=rnd)
    torch.cuda.synchronize()
    assert rd.status() == 0
    return w, rd, d, s


@pytest.mark.parametrize("name,over,use_ell", [
    ("tiny", {}, True),                                  # CUDA-core bias path, fp32
    ("tiny", {}, False),
    ("qwen3-8b", dict(R=5, gamma=4, V=2056, d=64), True),   # tensor cores, 17 tiles (ragged tail)
    ("deepseek-v4", dict(R=40, gamma=5, V=1288, d=64), False),  # bf16 logits, 200 rows = 2 row blocks
    ("stress", dict(R=24, gamma=6, V=4104, d=64), True),
])
def test_overlap_matches_oracle(name, over, use_ell):
    from speculative_decoding_draft_03_gb300 import binding as b
    w, rd, d, s = _round(name, 3, **over)
    ell = s["ell"] if use_ell else None
    if use_ell:
        # make sure both extremes of the length appear
        e = s["ell"].clone()
        e[0] = 0
        e[-1] = w["gamma"]
        ell = e
    got = b.acceptance_overlap(w["target"], w["U"], w["W1"], w["W2"], rd.x0, d["x"], d["lse"], ell,
                               w["temperature"])
    torch.cuda.synchronize()
    ref = oracle.acceptance_overlap(_host(w["target"]), _host(w["U"]), _host(w["W1"]), _host(w["W2"]),
                                    _host(rd.x0), _host(d["x"]), None if ell is None else _host(ell),
                                    w["temperature"])
    bf = any(w[k].dtype == torch.bfloat16 for k in ("U", "target", "W1", "W2"))
    _check(got.cpu().numpy(), ref, None if ell is None else _host(ell), 2e-3 if bf else 1e-5)


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),                                         # CUDA-core paths, fp32
    ("qwen3-8b", dict(R=5, gamma=4, V=2056, d=64)),       # tensor cores, ragged vocabulary tail
    ("deepseek-v4", dict(R=40, gamma=5, V=1288, d=64)),   # bf16 logits, 2 row blocks of positions
    ("stress", dict(R=24, gamma=6, V=4104, d=64)),
])
def test_verify_overlap_matches_verify_and_oracle(name, over):
    # dspark_verify_overlap: verification identical to dspark_verify, and the overlap of
    # every verified position equal to the oracle's (NaN past ell)
    from speculative_decoding_draft_03_gb300 import binding as b
    rnd = 6
    w, rd, d, s = _round(name, rnd, **over)
    ell = s["ell"].clone()
    ell[0] = 0
    ell[-1] = w["gamma"]
    args = (w["target"], w["U"], w["W1"], w["W2"], rd.x0, d["x"], d["logq"], d["lse"], ell, w["temperature"],
            w["req_id"], w["seed"], rnd)
    v1 = b.verify(*args)
    v2 = b.verify_overlap(*args)
    torch.cuda.synchronize()
    for k in ("n_acc", "tokens", "n_out"):
        assert torch.equal(v1[k], v2[k]), k
    ref = oracle.acceptance_overlap(_host(w["target"]), _host(w["U"]), _host(w["W1"]), _host(w["W2"]),
                                    _host(rd.x0), _host(d["x"]), _host(ell), w["temperature"])
    bf = any(w[k].dtype == torch.bfloat16 for k in ("U", "target", "W1", "W2"))
    _check(v2["overlap"].cpu().numpy(), ref, _host(ell), 2e-3 if bf else 1e-5)


def test_overlap_full_size_sampled_requests():
    from speculative_decoding_draft_03_gb300 import binding as b
    w, rd, d, s = _round("qwen3-8b", 5)
    got = b.acceptance_overlap(w["target"], w["U"], w["W1"], w["W2"], rd.x0, d["x"], d["lse"], s["ell"],
                               w["temperature"]).cpu().numpy()
    R = w["R"]
    rows = np.array(sorted({0, R // 2, R - 1}))
    idx = torch.from_numpy(rows).cuda()
    sub = {k: _host(w[k].index_select(0, idx)) for k in ("U", "target")}
    ell = _host(s["ell"])[rows]
    ref = oracle.acceptance_overlap(sub["target"], sub["U"], _host(w["W1"]), _host(w["W2"]), _host(rd.x0)[rows],
                                    _host(d["x"])[rows], ell, w["temperature"])
    _check(got[rows], ref, ell, 2e-3)


def test_overlap_bad_lengths_and_tokens_are_reported():
    from speculative_decoding_draft_03_gb300 import binding as b
    w, rd, d, s = _round("tiny", 1)
    R, gamma, V, rank = w["R"], w["gamma"], w["V"], w["rank"]
    for kind in ("ell", "token"):
        ws = b.workspace(b.acceptance_overlap_workspace_size(R, gamma, V, rank, w["W1"].dtype), w["U"].device)
        ell = torch.full((R,), gamma, dtype=torch.int32, device="cuda")
        x = d["x"].clone()
        if kind == "ell":
            ell[1] = gamma + 3
        else:
            x[2, 0] = V + 11
        out = b.acceptance_overlap(w["target"], w["U"], w["W1"], w["W2"], rd.x0, x, d["lse"], ell,
                                   w["temperature"], ws=ws)
        torch.cuda.synchronize()
        code = b.device_status(ws)
        assert code == 1, (kind, code)
        assert torch.isfinite(out).all()  # clamped: every position of every request evaluated
