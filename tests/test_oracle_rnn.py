"""Pins of the oracle's recurrent draft head (numb3r33 blog "RNN sequential head";
DSpark 精读 §2: a gated update of [s_{k-1}; E(x_{k-1}); h_k], bias W_o s_k).

Each special case reduces the head to something fixed elsewhere: with an identity
embedding path it is the Markov head (whose oracle is pinned separately); with the gate
shut the state stays at zero and the draft is softmax(U/T); with the gate open the cell is
a dense tanh layer; with a constant candidate the state follows the closed form of a
gated running average.  Sampling given the state is checked for its law.
"""
import math

import numpy as np
from scipy import special, stats

import oracle


def _bf16(a):
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _setup(R=3, gamma=4, V=48, ns=16, d=8, seed=0):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    h = rng.normal(0, 1, (R, gamma, d)).astype(np.float32)
    x0 = rng.integers(0, V, R)
    return rng, U, h, x0


def _conf(d, ns, rng):
    return rng.normal(0, 0.3, d + ns).astype(np.float32)


def test_identity_embedding_path_is_the_markov_head():
    # gate open (g = 1 exactly in binary64), candidate = tanh(E[x_{k-1}]) with E = atanh(W1):
    # s_k = W1[x_{k-1}] and the recurrent head draws exactly what the Markov head draws
    R, gamma, V, ns, d = 4, 5, 64, 16, 8
    rng, U, h, x0 = _setup(R, gamma, V, ns, d, seed=1)
    W1 = rng.uniform(-0.8, 0.8, (V, ns)).astype(np.float32)
    W2 = rng.normal(0, 0.6, (ns, V)).astype(np.float32)
    E = np.arctanh(W1.astype(np.float64)).astype(np.float32)
    Wse = np.zeros((2 * ns, 2 * ns), np.float32)
    Wse[ns:, ns:] = np.eye(ns)
    Wh = np.zeros((d, 2 * ns), np.float32)
    bgc = np.concatenate([np.full(ns, 60.0), np.zeros(ns)]).astype(np.float32)
    conf_w = _conf(d, ns, rng)
    temp = np.array([1.0, 0.9, 1.1, 1.2, 0.8], np.float32)
    rn = oracle.rnn_draft(U, E, Wse, Wh, bgc, W2, h, conf_w, 0.1, 1.3, temp, 0.7, x0, np.arange(R), 5, 2)
    mk = oracle.markov_draft(U, W1, W2, h, conf_w, 0.1, 1.3, temp, 0.7, x0, np.arange(R), 5, 2)
    # the stored state is W1[x_{k-1}] up to one fp32 rounding of tanh(atanh(.))
    for r in range(R):
        prev = [x0[r]] + list(mk["x"][r, :-1])
        np.testing.assert_allclose(rn["state"][r], W1[prev].astype(np.float64), rtol=3e-7, atol=0)
    assert (mk["margin"] > 1e-5).all()
    np.testing.assert_array_equal(rn["x"], mk["x"])
    np.testing.assert_allclose(rn["logq"], mk["logq"], atol=1e-5)
    np.testing.assert_allclose(rn["lse"], mk["lse"], atol=1e-5)
    np.testing.assert_allclose(rn["conf"], mk["conf"], atol=1e-6)


def test_shut_gate_keeps_the_zero_state():
    R, gamma, V, ns, d = 3, 4, 40, 8, 8
    rng, U, h, x0 = _setup(R, gamma, V, ns, d, seed=2)
    E = rng.normal(0, 1, (V, 8)).astype(np.float32)
    Wse = rng.normal(0, 1, (ns + 8, 2 * ns)).astype(np.float32)
    Wh = rng.normal(0, 1, (d, 2 * ns)).astype(np.float32)
    Wse[:, :ns] = 0
    Wh[:, :ns] = 0
    bgc = np.concatenate([np.full(ns, -60.0), rng.normal(0, 1, ns)]).astype(np.float32)
    Wo = rng.normal(0, 1, (ns, V)).astype(np.float32)
    conf_w = _conf(d, ns, rng)
    rn = oracle.rnn_draft(U, E, Wse, Wh, bgc, Wo, h, conf_w, 0.0, 1.0, np.ones(gamma, np.float32), 1.0, x0,
                          np.arange(R), 9, 0)
    assert np.abs(rn["state"]).max() < 1e-20
    zeros = np.zeros((V, 1), np.float32)
    mk = oracle.markov_draft(U, zeros, np.zeros((1, V), np.float32), h, np.zeros(d + 1, np.float32), 0.0, 1.0,
                             np.ones(gamma, np.float32), 1.0, x0, np.arange(R), 9, 0)
    np.testing.assert_array_equal(rn["x"], mk["x"])
    for r in range(R):
        for k in range(gamma):
            np.testing.assert_allclose(rn["lse"][r, k], special.logsumexp(U[r, k].astype(np.float64)), atol=1e-12)


def test_open_gate_is_a_dense_tanh_layer_on_the_hidden_state():
    # s_k = tanh(h_k Wh[:, ns:] + b_c), rounded to bf16 (bf16 weights): position k reads h row k-1
    R, gamma, V, ns, d = 2, 3, 32, 8, 12
    rng, U, h, x0 = _setup(R, gamma, V, ns, d, seed=3)
    E = _bf16(rng.normal(0, 1, (V, 4)))
    Wse = _bf16(np.zeros((ns + 4, 2 * ns)))
    Wh = _bf16(rng.normal(0, 0.4, (d, 2 * ns)))
    bc = rng.normal(0, 0.3, ns)
    bgc = np.concatenate([np.full(ns, 60.0), bc]).astype(np.float32)
    Wo = _bf16(rng.normal(0, 0.3, (ns, V)))
    rn = oracle.rnn_draft(U, E, Wse, Wh, bgc, Wo, h, _conf(d, ns, rng), 0.0, 1.0, np.ones(gamma, np.float32), 1.0,
                          x0, np.arange(R), 1, 0)
    wh = _bf16_to_f64(Wh)
    for r in range(R):
        for k in range(gamma):
            ref = np.tanh(h[r, k].astype(np.float64) @ wh[:, ns:] + bgc[ns:].astype(np.float64))
            # bf16 keeps 8 significant bits: half an ulp is at most 2^-8 of the value
            np.testing.assert_allclose(rn["state"][r, k], ref, rtol=2.0 ** -8, atol=0)
            assert np.array_equal(rn["state"][r, k], _bf16_to_f64(_bf16(rn["state"][r, k])))


def test_constant_candidate_gives_the_gated_running_average():
    # candidate tanh(b_c) at every position, gate from h only:
    # s_k = tanh(b_c) * (1 - prod_{i<=k} (1 - g_i)),  g_i = sigmoid(h_i Wh[:, :ns] + b_g)
    R, gamma, V, ns, d = 2, 6, 16, 4, 6
    rng, U, h, x0 = _setup(R, gamma, V, ns, d, seed=4)
    E = rng.normal(0, 1, (V, 3)).astype(np.float32)
    Wse = np.zeros((ns + 3, 2 * ns), np.float32)
    Wh = np.zeros((d, 2 * ns), np.float32)
    Wh[:, :ns] = rng.normal(0, 0.5, (d, ns))
    bgc = rng.normal(0, 0.5, 2 * ns).astype(np.float32)
    Wo = rng.normal(0, 0.3, (ns, V)).astype(np.float32)
    rn = oracle.rnn_draft(U, E, Wse, Wh, bgc, Wo, h, _conf(d, ns, rng), 0.0, 1.0, np.ones(gamma, np.float32), 1.0,
                          x0, np.arange(R), 3, 0)
    c = np.tanh(bgc[ns:].astype(np.float64))
    for r in range(R):
        keep = np.ones(ns)
        for k in range(gamma):
            g = special.expit(h[r, k].astype(np.float64) @ Wh[:, :ns].astype(np.float64) + bgc[:ns])
            keep *= 1.0 - g
            np.testing.assert_allclose(rn["state"][r, k], c * (1.0 - keep), rtol=2e-6, atol=1e-7)


def test_draw_given_the_state_follows_the_softmax():
    # position 1 of many requests with the same inputs: x_1 ~ softmax((U_1 + s_1 W_o)/T)
    N, V, ns, d, T = 200_000, 8, 4, 3, 0.8
    rng = np.random.default_rng(6)
    U = np.broadcast_to(rng.normal(0, 1, (1, 1, V)).astype(np.float32), (N, 1, V)).copy()
    h = np.broadcast_to(rng.normal(0, 1, (1, 1, d)).astype(np.float32), (N, 1, d)).copy()
    E = rng.normal(0, 1, (V, 2)).astype(np.float32)
    Wse = rng.normal(0, 0.5, (ns + 2, 2 * ns)).astype(np.float32)
    Wh = rng.normal(0, 0.5, (d, 2 * ns)).astype(np.float32)
    bgc = rng.normal(0, 0.5, 2 * ns).astype(np.float32)
    Wo = rng.normal(0, 1.0, (ns, V)).astype(np.float32)
    rn = oracle.rnn_draft(U, E, Wse, Wh, bgc, Wo, h, _conf(d, ns, rng), 0.0, 1.0, [1.0], T, np.full(N, 3),
                          np.arange(N), 12, 0)
    s1 = rn["state"][0, 0]
    assert (rn["state"][:, 0] == s1).all()
    p = special.softmax((U[0, 0].astype(np.float64) + s1 @ Wo.astype(np.float64)) / T)
    cnt = np.bincount(rn["x"][:, 0], minlength=V)
    assert stats.chisquare(cnt, p * N).pvalue > 1e-5
    np.testing.assert_allclose(rn["logq"][0, 0], math.log(p[rn["x"][0, 0]]), atol=1e-12)


def test_verify_with_state_rows_equals_verify_with_the_factor_rows():
    # the residual recomputation with explicit state rows W1[x_{j-1}] is the Markov one
    R, gamma, V, rank = 6, 3, 40, 8
    rng = np.random.default_rng(7)
    U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
    target = (np.concatenate([U, U[:, -1:]], 1) + rng.normal(0, 1.5, (R, gamma + 1, V))).astype(np.float32)
    W1 = rng.normal(0, 0.5, (V, rank)).astype(np.float32)
    W2 = rng.normal(0, 0.5, (rank, V)).astype(np.float32)
    x0 = rng.integers(0, V, R)
    d = oracle.markov_draft(U, W1, W2, np.zeros((R, gamma, 1), np.float32), np.zeros(1 + rank, np.float32), 0.0,
                            1.0, np.ones(gamma, np.float32), 1.0, x0, np.arange(R), 4, 1)
    prev = np.concatenate([x0[:, None], d["x"][:, :-1]], 1)
    state = W1[prev].astype(np.float64)
    ell = np.full(R, gamma, np.int32)
    a = oracle.verify(target, U, W1, W2, x0, d["x"], d["logq"], d["lse"], ell, 1.0, np.arange(R), 4, 1)
    b = oracle.verify(target, U, np.zeros((1, 1), np.float32), W2, x0, d["x"], d["logq"], d["lse"], ell, 1.0,
                      np.arange(R), 4, 1, state=state)
    assert (a["n_acc"] < gamma).any()  # some residual draws happen
    for k in ("n_acc", "tokens", "n_out", "corr_kind"):
        np.testing.assert_array_equal(a[k], b[k])


def test_confidence_for_given_states_matches_the_chain():
    R, gamma, V, ns, d = 3, 4, 32, 8, 5
    rng, U, h, x0 = _setup(R, gamma, V, ns, d, seed=8)
    E = rng.normal(0, 1, (V, 4)).astype(np.float32)
    Wse = rng.normal(0, 0.5, (ns + 4, 2 * ns)).astype(np.float32)
    Wh = rng.normal(0, 0.5, (d, 2 * ns)).astype(np.float32)
    bgc = rng.normal(0, 0.5, 2 * ns).astype(np.float32)
    Wo = rng.normal(0, 0.3, (ns, V)).astype(np.float32)
    conf_w = _conf(d, ns, rng)
    temp = rng.uniform(0.5, 1.5, gamma).astype(np.float32)
    rn = oracle.rnn_draft(U, E, Wse, Wh, bgc, Wo, h, conf_w, 0.2, 1.5, temp, 1.0, x0, np.arange(R), 3, 0)
    c = oracle.rnn_confidence(h, rn["state"], conf_w, 0.2, 1.5, temp)
    np.testing.assert_allclose(c, rn["conf"], rtol=0, atol=1e-15)
    # a zero state leaves the hidden-state part only: sigmoid(kappa (w_h . h + b) / T_k)
    c0 = oracle.rnn_confidence(h, np.zeros_like(rn["state"]), conf_w, 0.2, 1.5, temp)
    ref = special.expit(1.5 * (h.astype(np.float64) @ conf_w[:d].astype(np.float64) + 0.2) / temp)
    np.testing.assert_allclose(c0, ref, rtol=1e-12)
