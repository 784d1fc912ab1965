"""The core pin: the emitted tokens follow the target law.

(1) Exact enumeration (test-side, independent of the oracle) over every draft path at
    V=8, gamma=3: with the early-stop scheduler the law of each emitted y_m, given the
    earlier emitted tokens and that the round emitted at least m tokens, is the target
    row softmax(t_{m-1}/T) -- the exactness theorem of speculative sampling with the
    (p-q)+ residual and the bonus token.
(2) The oracle over 10^6 seeded trials matches that law (chi-square), for the early-
    stop and capacity-K schedulers and a non-unit temperature; its first-position
    acceptance rate equals 1 - TV(p, q) (binomial z-test).
"""
import itertools
import math

import numpy as np
import pytest
from scipy import special, stats

import oracle

V, GAMMA, RANK, D = 8, 3, 4, 5


def _problem(seed, T=1.0):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 1.2, (GAMMA, V)).astype(np.float32)
    W1 = rng.normal(0, 0.6, (V, RANK)).astype(np.float32)
    W2 = rng.normal(0, 0.6, (RANK, V)).astype(np.float32)
    target = np.concatenate([U, U[-1:]], 0) + rng.normal(0, 0.9, (GAMMA + 1, V)).astype(np.float32)
    target = target.astype(np.float32)
    h = rng.normal(0, 1, (GAMMA, D)).astype(np.float32)
    cw = rng.normal(0, 0.8, D + RANK).astype(np.float32)
    return dict(U=U, W1=W1, W2=W2, target=target, h=h, cw=cw, T=T, x0=3)


def _np_draft_law(P, x_prev, k):
    z = (P["U"][k].astype(np.float64) + P["W1"][x_prev].astype(np.float64) @ P["W2"].astype(np.float64)) / P["T"]
    return special.softmax(z)


def _np_conf(P, x_prev, k):
    d = D
    s = P["cw"][:d].astype(np.float64) @ P["h"][k].astype(np.float64) + \
        P["cw"][d:].astype(np.float64) @ P["W1"][x_prev].astype(np.float64)
    return np.float32(special.expit(s))


def _early_stop_len(conf, sps):
    # one request: the chain order is depth order; stop at the first non-increase
    a = np.cumprod(np.asarray(conf, np.float64))
    tau, n = 1.0, 0
    while n < len(a):
        if (tau + a[n]) * sps[2 + n] <= tau * sps[1 + n]:
            break
        tau += a[n]
        n += 1
    return n


def _exact_output_law(P, sps):
    """P(output sequence) by enumerating draft paths, scheduler decisions, accept/reject."""
    p_t = [special.softmax(P["target"][m].astype(np.float64) / P["T"]) for m in range(GAMMA + 1)]
    law = {}
    for path in itertools.product(range(V), repeat=GAMMA):
        prev, pq, qs, cs = P["x0"], 1.0, [], []
        for k in range(GAMMA):
            q = _np_draft_law(P, prev, k)
            cs.append(_np_conf(P, prev, k))
            qs.append(q)
            pq *= q[path[k]]
            prev = path[k]
        ell = _early_stop_len(cs, sps)
        alive = pq
        for j in range(ell + 1):
            if j == ell:  # every verified draft accepted: bonus from target row ell
                for y in range(V):
                    key = path[:j] + (y,)
                    law[key] = law.get(key, 0.0) + alive * p_t[j][y]
                break
            x = path[j]
            acc = min(1.0, p_t[j][x] / qs[j][x])
            rho = np.maximum(p_t[j] - qs[j], 0.0)
            if rho.sum() > 0:
                for y in range(V):
                    key = path[:j] + (y,)
                    law[key] = law.get(key, 0.0) + alive * (1 - acc) * rho[y] / rho.sum()
            alive *= acc
    return law, p_t


def test_exact_enumeration_reproduces_target_law():
    P = _problem(0)
    sps = 100.0 / (1.0 + np.arange(GAMMA + 2) / 8.0)
    law, p_t = _exact_output_law(P, sps)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    # conditional law of y_m given the emitted prefix and n >= m
    covered = 0
    for m in range(1, GAMMA + 2):
        prefixes = {}
        for seq, pr in law.items():
            if len(seq) >= m:
                prefixes.setdefault(seq[:m - 1], np.zeros(V))[seq[m - 1]] += pr
        covered += bool(prefixes)
        for pre, vec in prefixes.items():
            if vec.sum() > 1e-14:
                np.testing.assert_allclose(vec / vec.sum(), p_t[m - 1], atol=1e-10)
    assert covered >= 3  # the scheduler admits up to at least two drafts on some paths


def _oracle_trials(P, sps, mode, N, R, seed, hist=None):
    nb = N // R
    n = nb * R
    U = np.broadcast_to(P["U"], (n, GAMMA, V)).copy()
    h = np.broadcast_to(P["h"], (n, GAMMA, D)).copy()
    target = np.broadcast_to(P["target"], (n, GAMMA + 1, V)).copy()
    ids = np.arange(n, dtype=np.int64)
    x0 = np.full(n, P["x0"], np.int32)
    d = oracle.markov_draft(U, P["W1"], P["W2"], h, P["cw"], 0.0, 1.0, np.ones(GAMMA), P["T"], x0, ids, seed, 5)
    conf = d["conf"].astype(np.float32).reshape(nb, R, GAMMA)
    ell = oracle.schedule_many(conf, sps, mode, hist, 0).reshape(n)
    v = oracle.verify(target, U, P["W1"], P["W2"], x0, d["x"], d["logq"].astype(np.float32),
                      d["lse"].astype(np.float32), ell, P["T"], ids, seed, 5)
    return d, ell, v


def _check_law(v, p_t, N):
    toks, nout = v["tokens"], v["n_out"]
    for m in range(1, GAMMA + 2):
        sel = nout >= m
        cnt = np.bincount(toks[sel, m - 1], minlength=V)
        if sel.sum() < 2000:
            continue
        assert stats.chisquare(cnt, p_t[m - 1] * sel.sum()).pvalue > 1e-5, m
    # y_2 independent of y_1 given n >= 2 (context-free target): contingency vs marginal x p_t[1]
    sel = nout >= 2
    tab = np.zeros((V, V))
    np.add.at(tab, (toks[sel, 0], toks[sel, 1]), 1)
    rows = tab.sum(1)
    exp = np.outer(rows, p_t[1])
    keep = exp > 5
    chi = ((tab - exp)[keep] ** 2 / exp[keep]).sum()
    dof = keep.sum() - (rows > 0).sum()
    assert stats.chi2.sf(chi, dof) > 1e-5


@pytest.mark.parametrize("mode,T", [(oracle.EARLY_STOP, 1.0), (oracle.CAPACITY_K, 1.0),
                                    (oracle.EARLY_STOP, 0.7), (oracle.FIXED, 1.0)])
def test_oracle_emits_target_law_1e6_trials(mode, T):
    P = _problem(1, T)
    R = 2
    sps = 100.0 / (1.0 + np.arange(R * (GAMMA + 1) + 1) / 50.0)
    N = 1_000_000
    hist = None
    if mode == oracle.CAPACITY_K:
        rng = np.random.default_rng(9)
        hist = rng.uniform(0.2, 1.0, (N // R, R, GAMMA)).astype(np.float32)
    if mode == oracle.FIXED:
        d, ell, v = None, None, None
        nb = N // R
        n = nb * R
        U = np.broadcast_to(P["U"], (n, GAMMA, V)).copy()
        h = np.broadcast_to(P["h"], (n, GAMMA, D)).copy()
        target = np.broadcast_to(P["target"], (n, GAMMA + 1, V)).copy()
        ids = np.arange(n, dtype=np.int64)
        x0 = np.full(n, P["x0"], np.int32)
        d = oracle.markov_draft(U, P["W1"], P["W2"], h, P["cw"], 0.0, 1.0, np.ones(GAMMA), T, x0, ids, 17, 2)
        ell = np.full(n, GAMMA, np.int32)
        v = oracle.verify(target, U, P["W1"], P["W2"], x0, d["x"], d["logq"].astype(np.float32),
                          d["lse"].astype(np.float32), ell, T, ids, 17, 2)
        # first-position acceptance = sum min(p, q) = 1 - TV
        q1 = _np_draft_law(P, P["x0"], 0)
        p1 = special.softmax(P["target"][0].astype(np.float64) / T)
        alpha = np.minimum(p1, q1).sum()
        assert abs(alpha - (1 - 0.5 * np.abs(p1 - q1).sum())) < 1e-14
        rate = (v["n_acc"] >= 1).mean()
        assert abs(rate - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / n)
    else:
        d, ell, v = _oracle_trials(P, sps, mode, N, R, seed=3, hist=hist)
        assert (ell >= 0).all() and (ell <= GAMMA).all()
        assert len(np.unique(ell)) > 1  # the scheduler actually varies the length
    p_t = [special.softmax(P["target"][m].astype(np.float64) / T) for m in range(GAMMA + 1)]
    _check_law(v, p_t, N)
    # round bookkeeping: tokens = accepted drafts then one correction/bonus
    n_acc = v["n_acc"]
    assert (v["n_out"] == n_acc + 1).all()
    for j in range(GAMMA):
        sel = n_acc > j
        assert (v["tokens"][sel, j] == d["x"][sel, j]).all()
