"""Comparison rules between the CUDA path and the fp64 oracle.

* Token ids, accepted lengths and verify lengths match exactly, except a *boundary
  case*: the oracle's decision margin lies within 1e-5 (Gumbel key margin between the
  winner and the runner-up, |u - p/q| for an acceptance test, the relative Theta gap or
  the a-gap at the scheduler's cut, or a residual whose winner/runner-up has
  rho < 1e-3 max(p, q)).  A boundary case must also be consistent (the GPU picked the
  oracle's runner-up).  Boundary cases are counted; after one, the request's later
  positions are not compared (its path has legitimately diverged).
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
