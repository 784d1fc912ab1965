"""Comparison rules between the CUDA path and the fp64 oracle.

* Token ids, accepted lengths and verify lengths match exactly, except a *boundary
  case*: the oracle's decision margin lies within 1e-5 (Gumbel key margin between the
  winner and the runner-up, |u - p/q| for an acceptance test, the relative Theta gap or
  the a-gap at the scheduler's cut, or a residual whose winner/runner-up has
  rho < 1e-3 max(p, q)).  A boundary case must also be consistent (the GPU picked the
  oracle's runner-up).  Boundary cases are counted.  compare_draft stops comparing the
  request after one (its path has legitimately diverged); compare_draft_continuing lets
  the oracle adopt the GPU's token and keeps comparing the later positions.
* Probabilities and confidences: |gpu - ref| <= tol * max(|ref|, floor), tol = 1e-5
  where W1/W2 and the logits are fp32, 2e-3 where any of them is bf16; floor = 1 for
  log-domain values (logq, lse) and 1e-12 for confidences.
"""
from __future__ import annotations

import numpy as np

BOUNDARY = 1e-5
RHO_CANCEL = 1e-3


class Tally:
    def __init__(self):
        self.draws = 0
        self.boundary = 0
        self.notes = []

    def check_rate(self):
        allowed = max(1, int(1e-4 * self.draws))
        assert self.boundary <= allowed, (self.boundary, self.draws, self.notes[:5])


def close(gpu, ref, tol, floor):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    lim = tol * np.maximum(np.abs(ref), floor)
    bad = ~(err <= lim)
    return bad


def compare_draft(gpu, ref, tol, tally: Tally, rows=None):
    """gpu: dict of numpy arrays [R,gamma] (x, logq, lse, conf); ref: oracle output for the
    same requests (rows selects the gpu rows that ref covers).  Returns the number of
    (r,k) positions compared exactly."""
    gx = gpu["x"] if rows is None else gpu["x"][rows]
    R, gamma = ref["x"].shape
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    compared = 0
    for r in range(R):
        for k in range(gamma):
            tally.draws += 1
            if gx[r, k] != ref["x"][r, k]:
                ok = ref["margin"][r, k] < BOUNDARY and gx[r, k] == ref["runner_up"][r, k]
                assert ok, f"draft token mismatch r={r} k={k+1}: gpu {gx[r,k]} oracle {ref['x'][r,k]} " \
                           f"(margin {ref['margin'][r,k]:.3g}, runner-up {ref['runner_up'][r,k]})"
                tally.boundary += 1
                tally.notes.append(("draft", r, k))
                # lse and the confidence of this position do not depend on the draw
                for key, fl in (("lse", 1.0), ("conf", 1e-12)):
                    bad = close(sel(gpu[key])[r, k], ref[key][r, k], tol, fl)
                    assert not bad, (key, r, k)
                break
            compared += 1
            for key, fl in (("logq", 1.0), ("lse", 1.0), ("conf", 1e-12)):
                g = sel(gpu[key])[r, k]
                if close(g, ref[key][r, k], tol, fl):
                    raise AssertionError(f"{key} r={r} k={k+1}: gpu {g!r} oracle {ref[key][r,k]!r} tol {tol}")
    return compared


def compare_schedule(gpu, ref, tally: Tally, tau_tol=1e-9):
    tally.draws += 1
    same = (np.array_equal(gpu["ell"], ref["ell"]) and int(gpu["B"]) == ref["B"])
    if not same:
        ok = ref["gap"] < BOUNDARY or ref["tie"] < BOUNDARY
        assert ok, f"schedule mismatch: B gpu {int(gpu['B'])} oracle {ref['B']} (gap {ref['gap']:.3g}, tie {ref['tie']:.3g})"
        tally.boundary += 1
        tally.notes.append(("schedule",))
        return False
    # identical confidences give tau equal up to summation order (binary64); confidences
    # that went through the two draft stages differ within the probability tolerance
    assert abs(float(gpu["tau"]) - ref["tau"]) <= tau_tol * max(1.0, abs(ref["tau"])), (float(gpu["tau"]), ref["tau"])
    return True


def compare_verify(gpu, ref, tally: Tally, rows=None):
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    n_acc, toks, n_out = sel(gpu["n_acc"]), sel(gpu["tokens"]), sel(gpu["n_out"])
    R = len(ref["n_acc"])
    for r in range(R):
        tally.draws += int(ref["n_acc"][r]) + 2
        if n_acc[r] != ref["n_acc"][r]:
            j = min(n_acc[r], ref["n_acc"][r])  # first acceptance test where they differ
            m = ref["acc_margin"][r, j]
            assert abs(m) < BOUNDARY, f"n_acc mismatch r={r}: gpu {n_acc[r]} oracle {ref['n_acc'][r]} (u - ratio {m:.3g})"
            tally.boundary += 1
            tally.notes.append(("accept", r))
            continue
        assert n_out[r] == ref["n_out"][r] == n_acc[r] + 1
        assert np.array_equal(toks[r, :n_acc[r]], ref["tokens"][r, :n_acc[r]])
        assert (toks[r, n_acc[r] + 1:] == -1).all()
        y_g, y_o = toks[r, n_acc[r]], ref["tokens"][r, n_acc[r]]
        if y_g != y_o:
            ok = ref["corr_margin"][r] < BOUNDARY or min(ref["corr_rho"][r]) < RHO_CANCEL
            assert ok, f"correction token mismatch r={r}: gpu {y_g} oracle {y_o} kind {ref['corr_kind'][r]} " \
                       f"(margin {ref['corr_margin'][r]:.3g}, rho {ref['corr_rho'][r]})"
            tally.boundary += 1
            tally.notes.append(("correction", r))


def _row_f64(W, x):
    """Row x of a host weight array (float32, or raw bf16 bits as uint16) in float64."""
    row = np.asarray(W[int(x)])
    if row.dtype == np.uint16:
        return (row.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return row.astype(np.float64)


def compare_draft_continuing(gpu, ref, host, tol, tally):
    """Like compare_draft, but a boundary case does not end the comparison of its request:
    the oracle adopts the GPU's token (a draw within 1e-5 of a decision boundary may go
    either way, so both tokens are correct) and recomputes the
    request's later positions from it, draw by draw (oracle.draft_row for the draw and
    oracle.rnn_confidence with the factor row W1[x_{k-1}] as the state for c_k, which is
    the Markov head's confidence), and those are compared too.

    gpu: numpy arrays x, logq, lse, conf [n, gamma]; ref: oracle.markov_draft on the same n
    requests; host: dict of the same requests' U [n,gamma,V], h [n,gamma,d], req_id [n]
    and the shared W1, W2, conf_w, conf_b, conf_logit_scale, conf_temp, temperature, seed,
    rnd.  Returns the number of positions compared exactly."""
    import oracle
    n, gamma = ref["x"].shape
    compared = 0
    for r in range(n):
        adopted = False
        for k in range(gamma):
            if adopted:
                xp = int(gpu["x"][r, k - 1])
                arow = _row_f64(host["W1"], xp)
                one = oracle.draft_row(host["U"][r, k], arow, host["W2"], host["temperature"], host["seed"],
                                       int(host["req_id"][r]), host["rnd"], k + 1)
                c = oracle.rnn_confidence(host["h"][r:r + 1, k:k + 1], arow.reshape(1, 1, -1), host["conf_w"],
                                          host["conf_b"], host["conf_logit_scale"],
                                          np.asarray(host["conf_temp"])[k:k + 1])[0, 0]
                cur = dict(x=one["x"], logq=one["logq"], lse=one["lse"], conf=c, margin=one["margin"],
                           runner_up=one["runner_up"])
            else:
                cur = {key: ref[key][r, k] for key in ("x", "logq", "lse", "conf", "margin", "runner_up")}
            tally.draws += 1
            gx = gpu["x"][r, k]
            keys = (("logq", 1.0), ("lse", 1.0), ("conf", 1e-12))
            if gx != cur["x"]:
                ok = cur["margin"] < BOUNDARY and gx == cur["runner_up"]
                assert ok, f"draft token mismatch r={r} k={k+1}: gpu {gx} oracle {cur['x']} " \
                           f"(margin {cur['margin']:.3g}, runner-up {cur['runner_up']})"
                tally.boundary += 1
                tally.notes.append(("draft", r, k))
                keys = (("lse", 1.0), ("conf", 1e-12))  # independent of the draw
                adopted = True
            else:
                compared += 1
            for key, fl in keys:
                if close(gpu[key][r, k], cur[key], tol, fl):
                    raise AssertionError(f"{key} r={r} k={k+1}: gpu {gpu[key][r, k]!r} oracle {cur[key]!r} tol {tol}")
    return compared


def check_round_stagewise(w, wn, d, s, v, rnd, x0, tally):
    """Every request of one GPU round (numpy outputs d, s, v of the draft, scheduler and
    verification) against the oracle, stage by stage: the draft with the oracle adopting
    the GPU's token after a boundary case, the scheduler on the GPU's confidences, and
    verification on the GPU's drafts and verify lengths.  w: the workload (device
    tensors, for the dtypes); wn: its host copy; x0: the anchors the round used."""
    import torch
    import oracle
    bf = any(w[k].dtype == torch.bfloat16 for k in ("U", "target", "W1", "W2"))
    tol = 2e-3 if bf else 1e-5
    ref_d = oracle.markov_draft(wn["U"], wn["W1"], wn["W2"], wn["h"], wn["conf_w"], wn["conf_b"],
                                wn["conf_logit_scale"], wn["conf_temp"], wn["temperature"], x0, wn["req_id"],
                                wn["seed"], rnd)
    host = dict(wn, rnd=rnd)
    compare_draft_continuing(d, ref_d, host, tol, tally)
    ref_s = oracle.schedule(d["conf"], wn["sps"], wn["mode"], wn.get("conf_hist"), wn.get("fixed_len", 0))
    same = compare_schedule(dict(ell=s["ell"], B=s["B"][0], tau=s["tau"][0]), ref_s, tally, tau_tol=1e-9)
    ref_v = oracle.verify(wn["target"], wn["U"], wn["W1"], wn["W2"], x0, d["x"], d["logq"], d["lse"], s["ell"],
                          wn["temperature"], wn["req_id"], wn["seed"], rnd)
    compare_verify(v, ref_v, tally)
    # every request's output is well formed
    assert ((v["n_acc"] >= 0) & (v["n_acc"] <= s["ell"])).all()
    assert (v["n_out"] == v["n_acc"] + 1).all()
    assert int(s["B"][0]) == w["R"] + int(s["ell"].sum())
    return same
