"""Pins of the oracle's acceptance-overlap diagnostic c*_j = sum_v min(q_j(v), p_j(v))
(numb3r33 blog, "Total variation label").

The diagnostic is checked against the value the page prints for its worked example,
against the total-variation form 1 - ||q - p||_1 / 2 built from independently computed
distributions, and against the acceptance rate of the oracle's own sampling procedure
(the page derives c* as the expectation of min(1, p/q) under the draft).
"""
import json
import math
import os

import numpy as np
from scipy import special

import oracle
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(a):
    """float32 -> raw bf16 bits (round to nearest even)."""
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_worked_example_value():
    # q = (.40, .35, .25), p = (.35, .40, .25): different argmax, overlap 0.95
    g = _golden("overlap.json")
    V = 3
    U = np.log(np.asarray(g["p_draft"], np.float64)).astype(np.float32).reshape(1, 1, V)
    target = np.stack([np.log(np.asarray(g["p_target"], np.float64)),
                       np.zeros(V)]).astype(np.float32).reshape(1, 2, V)
    W1 = np.zeros((V, 1), np.float32)
    W2 = np.zeros((1, V), np.float32)
    c = oracle.acceptance_overlap(target, U, W1, W2, np.zeros(1), np.zeros((1, 1)))
    assert abs(c[0, 0] - g["overlap"]) < 1e-6


def test_total_variation_form_with_bias_rows_and_temperature():
    # every position of a ragged batch against 1 - ||q - p||_1 / 2, with q built from the
    # explicit factor product W1[x_{j-1}] W2 (x_0 at j = 1) and p from target row j-1
    rng = np.random.default_rng(5)
    R, gamma, V, rank, T = 3, 4, 40, 8, 0.7
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    target = (np.concatenate([U, U[:, -1:]], axis=1) + rng.normal(0, 0.8, (R, gamma + 1, V))).astype(np.float32)
    W1 = _bf16(rng.normal(0, 0.3, (V, rank)))
    W2 = _bf16(rng.normal(0, 0.3, (rank, V)))
    x0 = rng.integers(0, V, R)
    x = rng.integers(0, V, (R, gamma))
    ell = np.array([4, 0, 2], np.int32)
    c = oracle.acceptance_overlap(target, U, W1, W2, x0, x, ell, T)
    w1, w2 = _bf16_to_f64(W1), _bf16_to_f64(W2)
    for r in range(R):
        for j in range(1, gamma + 1):
            if j > ell[r]:
                assert math.isnan(c[r, j - 1])
                continue
            xp = x0[r] if j == 1 else x[r, j - 2]
            q = special.softmax((U[r, j - 1].astype(np.float64) + w1[xp] @ w2) / T)
            p = special.softmax(target[r, j - 1].astype(np.float64) / T)
            assert abs(c[r, j - 1] - (1.0 - 0.5 * np.abs(q - p).sum())) < 1e-12
    # without ell every position is evaluated
    call = oracle.acceptance_overlap(target, U, W1, W2, x0, x, None, T)
    assert not np.isnan(call).any()
    np.testing.assert_array_equal(call[0], c[0])


def test_expected_acceptance_of_the_sampling_procedure():
    # c*_1 is the probability that the draft token of position 1 is accepted, c*_2 that of
    # position 2 once x_1 is fixed: position 1 is made a point mass on token a in both the
    # draft and the target, so x_1 = a is always drafted and accepted
    N, V, rank, T = 200_000, 12, 4, 1.3
    rng = np.random.default_rng(21)
    a = 7
    u1 = np.full(V, -40.0)
    u1[a] = 40.0
    u2 = rng.normal(0, 1.0, V)
    t2 = u2 + rng.normal(0, 1.2, V)
    U = np.broadcast_to(np.stack([u1, u2]).astype(np.float32), (N, 2, V)).copy()
    target = np.broadcast_to(np.stack([u1, t2, np.zeros(V)]).astype(np.float32), (N, 3, V)).copy()
    W1 = rng.normal(0, 0.5, (V, rank)).astype(np.float32)
    W2 = rng.normal(0, 0.5, (rank, V)).astype(np.float32)
    ids = np.arange(N)
    d = oracle.markov_draft(U, W1, W2, np.zeros((N, 2, 1), np.float32), np.zeros(1 + rank, np.float32), 0.0, 1.0,
                            [1.0, 1.0], T, np.zeros(N), ids, 17, 0)
    assert (d["x"][:, 0] == a).all()
    v = oracle.verify(target, U, W1, W2, np.zeros(N), d["x"], d["logq"], d["lse"], np.full(N, 2, np.int32), T,
                      ids, 17, 0)
    assert (v["n_acc"] >= 1).all()
    c = oracle.acceptance_overlap(target[:1], U[:1], W1, W2, np.zeros(1), d["x"][:1], None, T)
    assert abs(c[0, 0] - 1.0) < 1e-12
    rate = (v["n_acc"] == 2).mean()
    assert abs(rate - c[0, 1]) < 5 * math.sqrt(c[0, 1] * (1 - c[0, 1]) / N)


def test_special_cases():
    rng = np.random.default_rng(2)
    V, rank = 64, 4
    U = rng.normal(0, 2, (2, 1, V)).astype(np.float32)
    W1 = np.zeros((V, rank), np.float32)
    W2 = np.zeros((rank, V), np.float32)
    # identical laws: overlap 1
    same = np.concatenate([U, U], axis=1)
    c = oracle.acceptance_overlap(same, U, W1, W2, np.zeros(2), np.zeros((2, 1)))
    np.testing.assert_allclose(c, 1.0, atol=1e-12)
    # disjoint supports (up to e^-60): overlap 0
    u = np.full((1, 1, V), -30.0, np.float32)
    u[0, 0, 0] = 30.0
    t = np.full((1, 2, V), -30.0, np.float32)
    t[0, 0, 1] = 30.0
    c = oracle.acceptance_overlap(t, u, W1, W2, np.zeros(1), np.zeros((1, 1)))
    assert 0.0 <= c[0, 0] < 1e-20
    # always inside [0, 1]; ell = 0 evaluates nothing
    t = rng.normal(0, 3, (2, 2, V)).astype(np.float32)
    c = oracle.acceptance_overlap(t, U, W1, W2, np.zeros(2), np.zeros((2, 1)))
    assert ((c > 0) & (c < 1)).all()
    c = oracle.acceptance_overlap(t, U, W1, W2, np.zeros(2), np.zeros((2, 1)), np.zeros(2, np.int32))
    assert np.isnan(c).all()
