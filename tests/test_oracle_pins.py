"""Pins of the fp64 oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: a value printed on a
page (fixtures under tests/golden/), a published known-answer vector, a closed form, a
special case that reduces to a library routine (scipy), or an exact identity.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Counter-based generator
# ---------------------------------------------------------------------------
def test_philox_known_answer_vectors():
    kat = _golden("philox4x32_10_kat.json")
    for vec in kat["vectors"]:
        ctr = [int(x, 16) for x in vec["ctr"]]
        key = [int(x, 16) for x in vec["key"]]
        out = [int(x, 16) for x in vec["out"]]
        assert list(oracle.philox4x32_10(ctr, key)) == out


def test_counter_layout_and_lanes():
    # word v%4 of the block whose 4th counter word is v/4; request, round, stream and
    # position occupy the other counter words; the seed is the key.
    seed, rid, rnd, stream, pos = 0x1234_5678_9ABC_DEF0, 77, 5, 2, 9
    for v in (0, 1, 2, 3, 4, 7, 1023, 151935):
        blk = oracle.philox4x32_10([rid, rnd, (stream << 24) | pos, v // 4],
                                   [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.draw_bits(seed, rid, rnd, stream, pos, v // 4, v % 4) == blk[v % 4]


def test_uniform_mapping_exact_and_open_interval():
    for b in (0, 0xFF, 0x100, 0x7FFFFFFF, 0x80000000, 0xFFFFFF00, 0xFFFFFFFF):
        u = oracle.uniform(b)
        assert u == ((b >> 8) + 0.5) / 2**24
        # binary32 holds u exactly below 1/2 and 1-u exactly above: a single-precision
        # Gumbel can therefore take -ln u from u (lower half) or log1p(-(1-u)) (upper half)
        # without rounding the draw
        if u < 0.5:
            assert float(np.float32(u)) == u
        else:
            assert float(np.float32(1.0 - u)) == 1.0 - u
        assert 0.0 < u < 1.0
    assert oracle.uniform(0) == 2.0**-25
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0**-25


def test_gumbel_tail_accuracy():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    for b in (0, 1 << 8, 0x80000000, 0xFFFFFE00, 0xFFFFFF00, 0xFFFFFFFF):
        u = oracle.uniform(b)
        exact = float(-mp.log(-mp.log(mp.mpf(u))))
        got = oracle.gumbel(u)
        assert abs(got - exact) <= 1e-14 * max(1.0, abs(exact))
    # largest possible draw: -ln(-ln(1 - 2^-25)) ~ 25 ln 2
    assert abs(oracle.gumbel(1 - 2.0**-25) - 25 * math.log(2)) < 1e-6


# ---------------------------------------------------------------------------
# Draft stage: special cases that reduce to library routines
# ---------------------------------------------------------------------------
def _draft_inputs(R, gamma, V, rank, d, rng, w_scale=0.5):
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    W1 = rng.normal(0, w_scale, (V, rank)).astype(np.float32)
    W2 = rng.normal(0, w_scale, (rank, V)).astype(np.float32)
    h = rng.normal(0, 1, (R, gamma, d)).astype(np.float32)
    cw = rng.normal(0, 0.3, d + rank).astype(np.float32)
    return U, W1, W2, h, cw


def test_draft_with_zero_bias_is_softmax_of_U():
    rng = np.random.default_rng(1)
    V = 37
    U, W1, W2, h, cw = _draft_inputs(1, 1, V, 4, 3, rng)
    W1[:] = 0
    for T in (1.0, 0.6):
        q = oracle.draft_distribution(U[0, 0], W1, W2, 3, T)
        np.testing.assert_allclose(q, special.softmax(U[0, 0].astype(np.float64) / T), rtol=1e-13)


def test_draft_identity_factor_reduces_to_transition_table():
    # rank = V and W1 = I: B = W1 W2 = W2, so row x_prev of the bias is W2[x_prev, :]
    # (a row, not a column: a transposed factor fails this on a non-symmetric table).
    rng = np.random.default_rng(2)
    V = 11
    U, _, _, h, cw = _draft_inputs(1, 1, V, V, 2, rng)
    W1 = np.eye(V, dtype=np.float32)
    table = rng.normal(0, 2.0, (V, V)).astype(np.float32)
    for x_prev in (0, 4, 10):
        q = oracle.draft_distribution(U[0, 0], W1, table, x_prev, 1.0)
        ref = special.softmax(U[0, 0].astype(np.float64) + table[x_prev].astype(np.float64))
        np.testing.assert_allclose(q, ref, rtol=1e-13)
        assert abs(q.sum() - 1.0) < 1e-14


def test_draft_outputs_normalise_and_logq_consistent():
    rng = np.random.default_rng(3)
    R, gamma, V, rank, d = 3, 4, 50, 6, 5
    U, W1, W2, h, cw = _draft_inputs(R, gamma, V, rank, d, rng)
    x0 = np.array([1, 7, 49], np.int32)
    out = oracle.markov_draft(U, W1, W2, h, cw, 0.0, 1.0, np.ones(gamma), 1.0, x0,
                              np.arange(R), 0, 0)
    for r in range(R):
        prev = x0[r]
        for k in range(gamma):
            q = oracle.draft_distribution(U[r, k], W1, W2, prev, 1.0)
            assert abs(q.sum() - 1.0) < 1e-13  # exact normalisation
            xk = out["x"][r, k]
            assert abs(out["logq"][r, k] - math.log(q[xk])) < 1e-12
            # lse: exp(z_x - lse) = q_x with z the unnormalised logit
            z = U[r, k].astype(np.float64) + W1[prev].astype(np.float64) @ W2.astype(np.float64)
            assert abs(out["lse"][r, k] - special.logsumexp(z)) < 1e-11
            prev = xk


def test_draft_bf16_inputs_are_exact_conversions():
    import torch
    rng = np.random.default_rng(4)
    R, gamma, V, rank, d = 2, 2, 40, 8, 4
    U, W1, W2, h, cw = _draft_inputs(R, gamma, V, rank, d, rng)
    as_bf = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    back = lambda t: t.to(torch.float32).numpy()
    Ub, W1b, W2b, hb = as_bf(U), as_bf(W1), as_bf(W2), as_bf(h)
    o_bf = oracle.markov_draft(bits(Ub), bits(W1b), bits(W2b), bits(hb), cw, 0.0, 1.0, np.ones(gamma),
                               1.0, np.array([0, 5]), np.arange(R), 9, 1)
    o_32 = oracle.markov_draft(back(Ub), back(W1b), back(W2b), back(hb), cw, 0.0, 1.0, np.ones(gamma),
                               1.0, np.array([0, 5]), np.arange(R), 9, 1)
    for k in ("x", "logq", "lse", "conf"):
        np.testing.assert_array_equal(o_bf[k], o_32[k])


def test_gumbel_max_draws_follow_softmax():
    # x_1 over many independent request ids ~ q_1 (chi-square, library softmax)
    rng = np.random.default_rng(5)
    V, rank, N = 8, 3, 200_000
    U1, W1, W2, _, _ = _draft_inputs(1, 1, V, rank, 1, rng)
    U = np.broadcast_to(U1, (N, 1, V)).copy()
    h = np.zeros((N, 1, 1), np.float32)
    out = oracle.markov_draft(U, W1, W2, h, np.zeros(1 + rank, np.float32), 0.0, 1.0, [1.0], 1.0,
                              np.full(N, 2), np.arange(N), 123, 0)
    q = special.softmax(U1[0, 0].astype(np.float64) + W1[2].astype(np.float64) @ W2.astype(np.float64))
    counts = np.bincount(out["x"][:, 0], minlength=V)
    assert stats.chisquare(counts, q * N).pvalue > 1e-5


def test_confidence_closed_forms():
    # c_k = sigmoid(kappa * (w_h.h_k + w_e.W1[x_{k-1}] + b) / T_k)
    V, rank, d, gamma = 6, 2, 3, 3
    U = np.zeros((1, gamma, V), np.float32)
    U[0, :, 4] = 30.0  # every draft token is 4 (q(4) ~ 1 - 5e-13)
    W1 = np.zeros((V, rank), np.float32)
    W1[2] = [1.0, 0.0]   # anchor row
    W1[4] = [0.0, 1.0]   # row of the sampled token 4
    W2 = np.zeros((rank, V), np.float32)
    h = np.ones((1, gamma, d), np.float32)
    ln3 = math.log(3.0)
    # w_h = 0, w_e picks row contents: position 1 sees W1[x0=2] -> logit ln3,
    # positions 2,3 see W1[4] -> logit 0 plus the bias b
    cw = np.array([0, 0, 0, ln3, 0.0], np.float32)
    out = oracle.markov_draft(U, W1, W2, h, cw, 0.0, 1.0, np.ones(gamma), 1.0, [2], [0], 0, 0)
    assert list(out["x"][0]) == [4, 4, 4]
    assert abs(out["conf"][0, 0] - 0.75) < 1e-7  # sigmoid(ln 3) = 3/4
    assert abs(out["conf"][0, 1] - 0.5) < 1e-15 and abs(out["conf"][0, 2] - 0.5) < 1e-15
    # bias b = ln 3 with kappa = 2 -> sigmoid(2 ln 3) = 9/10 at positions 2,3
    out = oracle.markov_draft(U, W1, W2, h, cw * 0, np.float32(ln3), 2.0, np.ones(gamma), 1.0, [2], [0], 0, 0)
    assert np.allclose(out["conf"][0], 0.9, atol=1e-7)
    # STS temperature T_k = 2: sigmoid(ln3 / 2) = sqrt3 / (1 + sqrt3)
    out = oracle.markov_draft(U, W1, W2, h, cw * 0, np.float32(ln3), 1.0, [2.0, 1.0, 1.0], 1.0, [2], [0], 0, 0)
    assert abs(out["conf"][0, 0] - math.sqrt(3) / (1 + math.sqrt(3))) < 1e-7
    assert abs(out["conf"][0, 1] - 0.75) < 1e-7
    # h-part: w_h = 1/d ones, h = ones -> w_h.h = 1
    cw_h = np.array([1 / 3, 1 / 3, 1 / 3, 0, 0], np.float32)
    out = oracle.markov_draft(U, W1, W2, h, cw_h, 0.0, 1.0, np.ones(gamma), 1.0, [2], [0], 0, 0)
    assert abs(out["conf"][0, 0] - special.expit(float(np.float64(np.float32(1 / 3)) * 3))) < 1e-15


# ---------------------------------------------------------------------------
# Verification: the pages' worked examples
# ---------------------------------------------------------------------------
def _one_position_trials(q, p, N, seed=7, temperature=1.0):
    """N independent one-token rounds with draft law q and target law p (fixed length 1)."""
    V = len(q)
    U = np.broadcast_to(np.log(np.asarray(q, np.float64)).astype(np.float32), (N, 1, V)).copy()
    target = np.broadcast_to(np.log(np.asarray(p, np.float64)).astype(np.float32), (N, 2, V)).copy()
    W1 = np.zeros((V, 1), np.float32)
    W2 = np.zeros((1, V), np.float32)
    h = np.zeros((N, 1, 1), np.float32)
    ids = np.arange(N)
    d = oracle.markov_draft(U, W1, W2, h, np.zeros(2, np.float32), 0.0, 1.0, [1.0], temperature,
                            np.zeros(N), ids, seed, 0)
    v = oracle.verify(target, U, W1, W2, np.zeros(N), d["x"], d["logq"], d["lse"], np.ones(N, np.int32),
                      temperature, ids, seed, 0)
    return d, v


def test_one_token_exactness_worked_example():
    g = _golden("one_token_exactness.json")
    N = 1_000_000
    d, v = _one_position_trials(g["q"], g["p"], N)
    acc = v["n_acc"] == 1
    # acceptance = sum min(p, q) = 0.8
    assert abs(acc.mean() - g["accept_total"]) < 5 * math.sqrt(0.16 / N)
    # accepted mass per token = min(p, q) = (0.4, 0.3, 0.1)
    joint = np.bincount(d["x"][acc, 0], minlength=3) / N
    np.testing.assert_allclose(joint, g["accepted_mass"], atol=5 * math.sqrt(0.25 / N))
    # residual draws follow (p-q)+ normalised = (0, 0.5, 0.5): token 0 never appears
    res = v["tokens"][~acc, 0]
    cnt = np.bincount(res, minlength=3)
    assert cnt[0] == 0
    assert stats.chisquare(cnt[1:], np.array(g["residual_normalised"][1:]) * len(res)).pvalue > 1e-5
    # emitted first token ~ p
    y = np.bincount(v["tokens"][:, 0], minlength=3)
    assert stats.chisquare(y, np.array(g["final"]) * N).pvalue > 1e-5


def test_overlap_worked_example():
    g = _golden("overlap.json")
    N = 1_000_000
    _, v = _one_position_trials(g["p_draft"], g["p_target"], N, seed=11)
    rate = (v["n_acc"] == 1).mean()
    assert abs(rate - g["overlap"]) < 5 * math.sqrt(0.95 * 0.05 / N)


def test_bonus_token_when_all_accepted_and_zero_length():
    # l = 0: the round still emits one token, drawn from target row 0 (bonus)
    N, V = 200_000, 5
    rng = np.random.default_rng(9)
    t = rng.normal(0, 1, V).astype(np.float32)
    target = np.broadcast_to(t, (N, 2, V)).copy()
    U = np.zeros((N, 1, V), np.float32)
    W1 = np.zeros((V, 1), np.float32)
    W2 = np.zeros((1, V), np.float32)
    v = oracle.verify(target, U, W1, W2, np.zeros(N), np.zeros((N, 1)), np.zeros((N, 1)), np.zeros((N, 1)),
                      np.zeros(N, np.int32), 1.0, np.arange(N), 3, 0)
    assert (v["n_acc"] == 0).all() and (v["n_out"] == 1).all() and (v["corr_kind"] == 0).all()
    cnt = np.bincount(v["tokens"][:, 0], minlength=V)
    assert stats.chisquare(cnt, special.softmax(t.astype(np.float64)) * N).pvalue > 1e-5
    assert (v["tokens"][:, 1] == -1).all()


def test_identical_laws_always_accept():
    # p == q: ratio 1 > u for every u in (0,1): every draft survives, bonus emitted
    _, v = _one_position_trials([0.2, 0.3, 0.5], [0.2, 0.3, 0.5], 50_000)
    assert (v["n_acc"] == 1).all() and (v["n_out"] == 2).all()
