"""Pins of the oracle's sequential temperature scaling (numb3r33 blog "Sequential
temperature scaling": calibrate position 1, freeze it, calibrate the cumulative survival
through position 2, and so on; mkdocs.reaper.mx "3 · DSpark" §3.2: a per-position
temperature search minimising the expected calibration error of prod_{i<=k} c_i).

* Held-out data drawn from a known law sigmoid(z_k / T*_k) give back T* at every
  position, which needs the frozen prefix and the survival outcome 1[L >= k].
* Logits that are all zero make every prediction 1/2: the ECE is |1/2 - mean outcome|
  at any temperature and the first grid point wins the tie.
* sigmoid(z/T) depends on z/T only: scaling the logits and the grid by the same factor
  scales the fitted temperatures by it and leaves the ECE unchanged.
* The sample order does not matter.
"""
import numpy as np

import oracle
from speculative_decoding_draft_03_gb300 import workloads as wl


def _data(N=40_000, T=(1.5, 0.7, 2.0, 1.0), seed=0):
    d = wl.sts_heldout(N, len(T), T, seed=seed)
    return d["z"].numpy(), d["acc_len"].numpy(), np.asarray(T)


def test_recovers_the_generating_temperatures():
    z, L, T = _data()
    grid = wl.sts_grid(128)
    Tf, ece = oracle.sts_fit(z, L, grid, 15)
    assert (np.abs(np.log(Tf) - np.log(T)) < 0.15).all(), (Tf, T)
    assert (ece < 0.02).all(), ece
    # the uncalibrated head (T = 1 everywhere) is measurably worse where T* is far from 1
    raw = [oracle.sts_ece(z, L, np.ones(k - 1), k, 1.0, 15) for k in (1, 2, 3)]
    assert raw[0] > 2 * ece[0] and raw[2] > 2 * ece[2]


def test_zero_logits_give_the_outcome_gap_and_the_first_grid_point():
    N, gamma = 1000, 2
    z = np.zeros((N, gamma), np.float32)
    L = np.zeros(N, np.int32)
    L[:300] = 2  # 30% survive both positions
    L[300:500] = 1
    grid = np.array([0.5, 1.0, 2.0, 4.0], np.float32)
    T, ece = oracle.sts_fit(z, L, grid, 10)
    np.testing.assert_array_equal(T, [0.5, 0.5])
    # position 1: p = 1/2, mean outcome 0.5 -> 0; position 2: p = 1/4, mean outcome 0.3
    np.testing.assert_allclose(ece, [0.0, 0.05], atol=1e-12)


def test_scale_equivariance_and_order_invariance():
    z, L, _ = _data(N=8000, seed=3)
    grid = wl.sts_grid(64)
    T1, e1 = oracle.sts_fit(z, L, grid, 15)
    T2, e2 = oracle.sts_fit(z * 4.0, L, grid * 4.0, 15)
    np.testing.assert_allclose(T2, 4.0 * T1, rtol=1e-6)
    np.testing.assert_allclose(e2, e1, rtol=1e-9, atol=1e-12)
    perm = np.random.default_rng(1).permutation(len(L))
    T3, e3 = oracle.sts_fit(z[perm], L[perm], grid, 15)
    np.testing.assert_array_equal(T3, T1)
    np.testing.assert_allclose(e3, e1, rtol=1e-9, atol=1e-12)
