"""dspark_verify_ragged: verification on a flattened target batch (each request's verify
rows packed at its own offset, in any order, with unused rows in between; numb3r33 blog
"Variable-length verification without wasting kernels") computes exactly what
dspark_verify computes on the padded [R, gamma+1, V] target, and what the fp64 oracle
computes on the padded target that the host rebuilds from the flattened rows and their
offsets."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_03_gb300 import workloads as wl
from tests.parity import Tally, compare_verify

pytestmark = pytest.mark.gpu


def _flatten(target, ell, rng):
    """Rows 0..ell[r] of each request, requests in a shuffled order, one unused row
    between consecutive requests."""
    R = target.shape[0]
    order = rng.permutation(R)
    rows, offsets, n = [], np.zeros(R, np.int32), 0
    for r in order:
        rows.append(torch.full_like(target[r, :1], float("nan")))  # an unused row, never read
        n += 1
        offsets[r] = n
        k = int(ell[r]) + 1
        rows.append(target[r, :k])
        n += k
    return torch.cat(rows, 0).contiguous(), torch.from_numpy(offsets).cuda()


def _host(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _unflatten(flat, offsets, ell, gamma):
    """[R, gamma+1, V] with request r's rows t = 0..ell[r] taken from flat[offsets[r] + t]
    (the rows past ell[r] are never read; they stay zero)."""
    R = len(offsets)
    out = np.zeros((R, gamma + 1, flat.shape[1]), flat.dtype)
    for r in range(R):
        n = int(ell[r]) + 1
        out[r, :n] = flat[offsets[r]:offsets[r] + n]
    return out


@pytest.mark.parametrize("name,over", [("tiny", {}), ("qwen3-8b", dict(V=20000, d=256)),
                                       ("deepseek-v4", dict(V=4104, d=256)), ("stress", dict(V=2056, d=64))])
def test_ragged_matches_padded(name, over):
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make(name, device="cuda", **over)
    rd = b.Round(w)
    rng = np.random.default_rng(7)
    tally = Tally()
    for rnd in (2, 3):
        d, s, v = rd.run(rnd=rnd)
        torch.cuda.synchronize()
        ref = {k: t.clone() for k, t in v.items()}
        ell = s["ell"].cpu().numpy()
        flat, off = _flatten(w["target"], ell, rng)
        got = b.verify_ragged(flat, off, w["U"], w["W1"], w["W2"], rd.x0, d["x"], d["logq"], d["lse"], s["ell"],
                              w["temperature"], w["req_id"], w["seed"], rnd)
        torch.cuda.synchronize()
        for k in ("n_acc", "tokens", "n_out"):
            assert torch.equal(got[k], ref[k]), (name, rnd, k)
        # the oracle on the padded target rebuilt on the host from the flattened rows
        padded = _unflatten(_host(flat), off.cpu().numpy(), ell, w["gamma"])
        ref_o = oracle.verify(padded, _host(w["U"]), _host(w["W1"]), _host(w["W2"]), _host(rd.x0), _host(d["x"]),
                              _host(d["logq"]), _host(d["lse"]), ell, w["temperature"], _host(w["req_id"]),
                              w["seed"], rnd)
        compare_verify({k: t.cpu().numpy() for k, t in got.items()}, ref_o, tally)
    tally.check_rate()


def test_ragged_offset_out_of_range_is_reported():
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make("tiny", device="cuda")
    rd = b.Round(w)
    d, s, v = rd.run(rnd=1)
    torch.cuda.synchronize()
    flat, off = _flatten(w["target"], s["ell"].cpu().numpy(), np.random.default_rng(0))
    off[2] = flat.shape[0] + 3
    R, gamma, V, rank = w["R"], w["gamma"], w["V"], w["rank"]
    ws = b.workspace(b.verify_workspace_size(R, gamma, V, rank, w["W1"].dtype), flat.device)
    b.verify_ragged(flat, off, w["U"], w["W1"], w["W2"], rd.x0, d["x"], d["logq"], d["lse"], s["ell"],
                    w["temperature"], w["req_id"], w["seed"], 1, ws=ws)
    torch.cuda.synchronize()
    assert b.device_status(ws, reset=True) == 1
