"""Pins of the oracle's confidence scheduler: the pages' examples, brute-force optimum
over every length vector on tiny instances, prefix closure, and each mode's rule."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _flat_then(R, gamma, flat_until, after):
    n = R * (gamma + 1) + 1
    sps = np.full(n, 100.0)
    sps[flat_until + 1:] = after
    return sps


def test_survival_stones_and_expected_length():
    g = _golden("survival.json")
    c = np.array([g["stones"]["c"]], np.float32)
    path = oracle.schedule_path(c, np.ones(6))
    np.testing.assert_allclose(np.round(path["a"], 2), g["stones"]["reach_printed_2dp"], atol=1e-12)
    assert abs(path["a"][2] - g["stones"]["reach_stone3_exact"]) < 1e-7
    # l = 4 fixed: tau = 1 + c1 + c1c2 + c1c2c3 + c1c2c3c4 (the page's expected output length)
    s = oracle.schedule(c, np.ones(6), oracle.FIXED, fixed_len=4)
    assert abs(s["tau"] - (1 + 0.9 + 0.72 + 0.504 + 0.1008)) < 1e-6
    assert s["B"] == 5 and list(s["ell"]) == [4]


def test_cumulative_and_calibration_products():
    g = _golden("survival.json")
    for key, exact in (("cumulative", "a5_exact"),):
        c = np.array([g[key]["c"]], np.float32)
        a = oracle.schedule_path(c, np.ones(len(g[key]["c"]) + 2))["a"]
        assert abs(a[-1] - g[key][exact]) < 1e-6
        assert abs(round(a[-1], 2) - g[key]["a5_printed_approx"]) < 1e-12
    cal = g["calibration"]
    a_raw = oracle.schedule_path(np.array([cal["raw_c"]], np.float32), np.ones(6))["a"]
    assert abs(a_raw[-1] - cal["raw_exact"]) < 1e-6 and round(a_raw[-1], 2) == cal["raw_printed_approx"]
    a_cal = oracle.schedule_path(np.array([cal["calibrated_c"]], np.float32), np.ones(6))["a"]
    assert abs(a_cal[-1] - cal["calibrated_exact"]) < 1e-6  # page prints 0.34 (slip), product is 0.3764


def test_greedy_order_and_cutoff_example():
    g = _golden("scheduler_examples.json")["greedy_order"]
    A, B = g["chains"]["A"], g["chains"]["B"]
    # conditional confidences reproducing the chains' cumulative survivals
    conf = np.array([[A[0], A[1] / A[0]], [B[0], B[1] / B[0]]], np.float32)
    path = oracle.schedule_path(conf, np.ones(7))
    names = [("A", "B")[r] + str(j) for r, j in zip(path["req"], path["depth"])]
    assert names == g["order"]
    # a step table that makes the fourth admission lower Theta: the cutoff falls before B2
    sps = np.array([100, 100, 100, 100, 100, 100, 90.0])
    s = oracle.schedule(conf, sps, oracle.EARLY_STOP)
    admitted = [f"A{j}" for j in range(1, s["ell"][0] + 1)] + [f"B{j}" for j in range(1, s["ell"][1] + 1)]
    assert sorted(admitted) == sorted(g["admitted"])
    assert s["B"] == 2 + 3
    assert abs(s["tau"] - (2 + A[0] + B[0] + A[1])) < 1e-6


def test_objective_table_decisions():
    g = _golden("scheduler_examples.json")["objective_table"]["rows"]
    for row in g:
        assert abs(row["tau"] * row["sps"] - row["theta"]) < 1e-9
    # One request with three certain drafts (a = 1,1,1: tau(3) = 4 with the guaranteed token);
    # the fourth draft's survival decides, with the table's step rates at B = 4 -> 5.
    for surv4, sps5, admit in ((0.8, 95.0, True), (0.2, 80.0, False)):
        conf = np.array([[1.0, 1.0, 1.0, surv4]], np.float32)
        sps = np.array([0, 100.0, 100.0, 100.0, 100.0, sps5])
        s = oracle.schedule(conf, sps, oracle.EARLY_STOP)
        assert (s["ell"][0] == 4) == admit
        # Theta compare: (4 + a4) * sps5 vs 4 * 100 -- the same comparison as the table's
        assert ((4 + np.float32(surv4)) * sps5 > 400) == admit


def _brute_force(conf, sps):
    R, gamma = conf.shape
    a = np.cumprod(conf.astype(np.float64), axis=1)
    best, best_l = -1.0, None
    for ell in itertools.product(range(gamma + 1), repeat=R):
        tau = R + sum(a[r, :ell[r]].sum() for r in range(R))
        B = R + sum(ell)
        th = tau * sps[B]
        if th > best + 1e-12:
            best, best_l = th, ell
    return best, best_l


def test_full_search_is_brute_force_optimum():
    rng = np.random.default_rng(0)
    for trial in range(300):
        R = int(rng.integers(1, 4))
        gamma = int(rng.integers(1, 4))
        conf = rng.uniform(0.05, 1.0, (R, gamma)).astype(np.float32)
        n = R * (gamma + 1) + 1
        kind = trial % 3
        if kind == 0:
            sps = 1000.0 / (1.0 + np.arange(n) / rng.uniform(1, 8))
        elif kind == 1:
            sps = 1000.0 * 0.8 ** np.floor(np.arange(n) / rng.integers(1, 4))
        else:
            sps = rng.uniform(10, 100, n)
        s = oracle.schedule(conf, sps, oracle.FULL_SEARCH)
        best, _ = _brute_force(conf, sps)
        assert abs(s["tau"] * sps[s["B"]] - best) <= 1e-9 * best


def test_early_stop_equals_full_search_on_hyperbolic_sps():
    # SPS(B) = S/(alpha + B): once a candidate fails to raise Theta no later one can
    rng = np.random.default_rng(1)
    for _ in range(200):
        R, gamma = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        conf = rng.uniform(0.01, 1.0, (R, gamma)).astype(np.float32)
        n = R * (gamma + 1) + 1
        sps = 1000.0 / (rng.uniform(0.5, 64) + np.arange(n))
        e = oracle.schedule(conf, sps, oracle.EARLY_STOP)
        f = oracle.schedule(conf, sps, oracle.FULL_SEARCH)
        assert e["B"] == f["B"] and (e["ell"] == f["ell"]).all()


def test_prefix_closure_including_exact_ties():
    rng = np.random.default_rng(2)
    for _ in range(200):
        R, gamma = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        conf = rng.uniform(0.0, 1.0, (R, gamma)).astype(np.float32)
        conf[rng.uniform(size=conf.shape) < 0.3] = 1.0  # equal a along chains
        conf[rng.uniform(size=conf.shape) < 0.05] = 0.0
        n = R * (gamma + 1) + 1
        sps = rng.uniform(10, 100, n)
        path = oracle.schedule_path(conf, sps)
        seen = set()
        for r, j in zip(path["req"], path["depth"]):
            assert j == 1 or (r, j - 1) in seen  # every prefix precedes its extension
            seen.add((r, j))
        for mode in (oracle.EARLY_STOP, oracle.FULL_SEARCH):
            s = oracle.schedule(conf, sps, mode)
            nstar = s["B"] - R
            adm = {}
            for r, j in zip(path["req"][:nstar], path["depth"][:nstar]):
                adm.setdefault(r, []).append(j)
            for r in range(R):
                assert sorted(adm.get(r, [])) == list(range(1, s["ell"][r] + 1))


def test_early_stop_rule_first_non_increase():
    rng = np.random.default_rng(3)
    for _ in range(200):
        R, gamma = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        conf = rng.uniform(0.0, 1.0, (R, gamma)).astype(np.float32)
        n = R * (gamma + 1) + 1
        sps = rng.uniform(10, 100, n)
        th = oracle.schedule_path(conf, sps)["theta"]
        s = oracle.schedule(conf, sps, oracle.EARLY_STOP)
        k = s["B"] - R
        assert all(th[i + 1] > th[i] for i in range(k))
        assert k == R * gamma or th[k + 1] <= th[k]
        assert abs(s["tau"] * sps[s["B"]] - th[k]) <= 1e-12 * th[k]


def test_capacity_k_counts_from_stale_confidences():
    rng = np.random.default_rng(4)
    for _ in range(100):
        R, gamma = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        conf = rng.uniform(0.0, 1.0, (R, gamma)).astype(np.float32)
        hist = rng.uniform(0.0, 1.0, (R, gamma)).astype(np.float32)
        n = R * (gamma + 1) + 1
        sps = 1000.0 * 0.85 ** np.floor(np.arange(n) / 3)
        K = oracle.schedule(hist, sps, oracle.FULL_SEARCH)["B"] - R
        s = oracle.schedule(conf, sps, oracle.CAPACITY_K, conf_hist=hist)
        assert s["B"] - R == min(K, R * gamma) == s["ell"].sum()
        # the admitted set is the top-K of the current order
        path = oracle.schedule_path(conf, sps)
        cnt = np.bincount(path["req"][:K], minlength=R)
        assert (cnt == s["ell"]).all()


def test_fixed_mode_and_zero_length():
    conf = np.full((3, 4), 0.5, np.float32)
    sps = np.ones(3 * 5 + 1)
    for L in (0, 2, 4, 9):
        s = oracle.schedule(conf, sps, oracle.FIXED, fixed_len=L)
        Le = min(L, 4)
        assert (s["ell"] == Le).all() and s["B"] == 3 * (1 + Le)
        assert abs(s["tau"] - 3 * (1 + sum(0.5 ** j for j in range(1, Le + 1)))) < 1e-12


def test_threshold_mode_worked_example():
    """Fixed confidence cutoff (vllmbangkok "Verify smarter, not longer"): each request keeps
    its leading drafts with c >= threshold; a token at exactly the cutoff is kept."""
    conf = np.array([[0.9, 0.8, 0.3],
                     [0.2, 0.95, 0.9],
                     [1.0, 1.0, 1.0],
                     [0.5, 0.5, 0.49]], np.float32)
    out = oracle.schedule_threshold(conf, 0.5)
    assert out["ell"].tolist() == [2, 0, 3, 2]
    assert out["B"] == 4 + 7
    a = lambda *c: np.cumprod(np.array(c, np.float64)).sum()
    tau = 4 + a(np.float32(0.9), np.float32(0.8)) + a(1.0, 1.0, 1.0) + a(0.5, 0.5)
    assert out["tau"] == pytest.approx(tau, rel=1e-15)
    # cutoffs above 1 keep nothing, cutoffs at or below 0 keep everything
    assert oracle.schedule_threshold(conf, 1.01)["ell"].tolist() == [0, 0, 0, 0]
    assert oracle.schedule_threshold(conf, 0.0)["ell"].tolist() == [3, 3, 3, 3]


def test_threshold_mode_is_prefix_closed_and_monotone():
    rng = np.random.default_rng(11)
    conf = rng.uniform(0, 1, (64, 9)).astype(np.float32)
    prev = None
    for th in (0.9, 0.7, 0.5, 0.3, 0.1):
        ell = oracle.schedule_threshold(conf, th)["ell"]
        for r in range(64):
            assert (conf[r, :ell[r]] >= th).all()
            assert ell[r] == 9 or conf[r, ell[r]] < th
        if prev is not None:
            assert (ell >= prev).all()  # lowering the cutoff never shortens a prefix
        prev = ell
