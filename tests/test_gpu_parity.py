"""CUDA path vs the fp64 oracle, stage by stage and for whole rounds.

Every GPU call goes through the C ABI (libdspark.so via the ctypes binding).  Inputs
are the seeded synthetic workloads; stage inputs handed to the GPU in the stage-wise
tests come from the oracle (never the reverse).  Sizes: the tiny workload in full, the
four large workloads at reduced vocabulary/hidden sizes that keep their distributions,
request counts and draft lengths (several vocabulary tiles plus a ragged tail), and --
in test_gpu_fullsize.py -- the full sizes on sampled requests.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_03_gb300 import workloads as wl
from tests.parity import Tally, check_round_stagewise, compare_draft, compare_schedule, compare_verify

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": {},
    "qwen3-8b": dict(V=20000, d=512),
    "batch128": dict(V=6000, d=256),
    "deepseek-v4": dict(V=4104, d=256),
    "stress": dict(V=2056, d=256),
}


def _b():
    from speculative_decoding_draft_03_gb300 import binding
    return binding


def _tol(w):
    bf = any(w[k].dtype == torch.bfloat16 for k in ("U", "target", "W1", "W2"))
    return 2e-3 if bf else 1e-5


def _np(d):
    return {k: v.detach().cpu().numpy() for k, v in d.items()}


def _gpu_workload(name, **over):
    w = wl.make(name, device="cpu", **over)
    wn = wl.to_numpy(w)
    wg = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    return wg, wn


def _oracle_draft(wn, rows=None, rnd=0, x0=None):
    src = wl.subset(wn, rows) if rows is not None else wn
    return oracle.markov_draft(src["U"], wn["W1"], wn["W2"], src["h"], wn["conf_w"], wn["conf_b"],
                               wn["conf_logit_scale"], wn["conf_temp"], wn["temperature"],
                               src["x0"] if x0 is None else x0, src["req_id"], wn["seed"], rnd)


@pytest.mark.parametrize("name", list(SMALL))
def test_draft_stage_matches_oracle(name):
    b = _b()
    wg, wn = _gpu_workload(name, **SMALL[name])
    d = b.markov_draft(wg["U"], wg["W1"], wg["W2"], wg["h"], wg["conf_w"], wg["conf_b"],
                       wg["conf_logit_scale"], wg["conf_temp"], wg["temperature"], wg["x0"], wg["req_id"],
                       wg["seed"], 3)
    torch.cuda.synchronize()
    ref = _oracle_draft(wn, rnd=3)
    tally = Tally()
    n = compare_draft(_np(d), ref, _tol(wg), tally)
    tally.check_rate()
    assert n >= 0.99 * wn["R"] * wn["gamma"] - tally.boundary * wn["gamma"]


@pytest.mark.parametrize("name", list(SMALL))
def test_schedule_stage_matches_oracle(name):
    b = _b()
    wg, wn = _gpu_workload(name, **SMALL[name])
    ref_d = _oracle_draft(wn)
    conf = ref_d["conf"].astype(np.float32)
    tally = Tally()
    for mode in (wl.EARLY_STOP, wl.FULL_SEARCH, wl.CAPACITY_K, wl.FIXED):
        hist = wn["conf_hist"] if wn["conf_hist"] is not None else \
            np.random.default_rng(5).uniform(0, 1, conf.shape).astype(np.float32)
        ref = oracle.schedule(conf, wn["sps"], mode, hist if mode == wl.CAPACITY_K else None, fixed_len=3)
        g = b.schedule(torch.from_numpy(conf).cuda(), wg["sps"], mode,
                       torch.from_numpy(hist).cuda() if mode == wl.CAPACITY_K else None, fixed_len=3)
        torch.cuda.synchronize()
        g = _np(g)
        compare_schedule(dict(ell=g["ell"], B=g["B"][0], tau=g["tau"][0]), ref, tally)
        ell = g["ell"]
        assert ell.min() >= 0 and ell.max() <= wn["gamma"]
    tally.check_rate()


@pytest.mark.parametrize("name", list(SMALL))
def test_verify_stage_matches_oracle(name):
    b = _b()
    wg, wn = _gpu_workload(name, **SMALL[name])
    ref_d = _oracle_draft(wn, rnd=1)
    R, gamma = wn["R"], wn["gamma"]
    rng = np.random.default_rng(11)
    ell = rng.integers(0, gamma + 1, R).astype(np.int32)  # every length, including 0 and gamma
    ell[:2] = [0, gamma]
    x = ref_d["x"]
    logq = ref_d["logq"].astype(np.float32)
    lse = ref_d["lse"].astype(np.float32)
    ref = oracle.verify(wn["target"], wn["U"], wn["W1"], wn["W2"], wn["x0"], x, logq, lse, ell,
                        wn["temperature"], wn["req_id"], wn["seed"], 1)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g = b.verify(wg["target"], wg["U"], wg["W1"], wg["W2"], wg["x0"], t(x), t(logq), t(lse), t(ell),
                 wg["temperature"], wg["req_id"], wg["seed"], 1)
    torch.cuda.synchronize()
    tally = Tally()
    compare_verify(_np(g), ref, tally)
    tally.check_rate()
    # the workload must exercise both corrections
    kinds = set(ref["corr_kind"].tolist())
    assert 0 in kinds and (1 in kinds or R < 8)


@pytest.mark.parametrize("name,over", [("qwen3-8b", dict(V=4104, d=64)), ("tiny", {})])
def test_residual_without_positive_mass_draws_from_p(name, over):
    """The residual's rounding fallback: with the draft normalisers handed in far too small,
    q exceeds p everywhere, so (p - q)+ is empty and every rejected request must be drawn
    from p with the residual's own random numbers (the oracle does the same); logq is made
    large so that the first draft is rejected."""
    b = _b()
    wg, wn = _gpu_workload(name, **over)
    ref_d = _oracle_draft(wn, rnd=1)
    R, gamma = wn["R"], wn["gamma"]
    ell = np.full(R, gamma, np.int32)
    x = ref_d["x"]
    logq = np.full((R, gamma), 50.0, np.float32)          # ratio p/q ~ e^-50: reject at j = 1
    lse = (ref_d["lse"] - 30.0).astype(np.float32)        # q = e^(z - lse) inflated by e^30
    ref = oracle.verify(wn["target"], wn["U"], wn["W1"], wn["W2"], wn["x0"], x, logq, lse, ell,
                        wn["temperature"], wn["req_id"], wn["seed"], 1)
    assert (ref["n_acc"] == 0).all()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g = b.verify(wg["target"], wg["U"], wg["W1"], wg["W2"], wg["x0"], t(x), t(logq), t(lse), t(ell),
                 wg["temperature"], wg["req_id"], wg["seed"], 1)
    torch.cuda.synchronize()
    tally = Tally()
    compare_verify(_np(g), ref, tally)
    tally.check_rate()


@pytest.mark.parametrize("name", list(SMALL))
def test_round_matches_oracle(name):
    """Whole round on the GPU (draft -> schedule -> verify chained on device) vs the
    oracle's round; exact unless a boundary case occurs (then stage-wise checks apply)."""
    b = _b()
    wg, wn = _gpu_workload(name, **SMALL[name])
    rd = b.Round(wg)
    d, s, v = rd.run(rnd=2)
    torch.cuda.synchronize()
    assert rd.status() == 0
    ref = oracle.run_round(wn, rnd=2)
    tally = Tally()
    compare_draft(_np(d), ref["draft"], _tol(wg), tally)
    if tally.boundary == 0:
        gs = _np(s)
        same = compare_schedule(dict(ell=gs["ell"], B=gs["B"][0], tau=gs["tau"][0]), ref["sched"], tally,
                                _tol(wg))
        if same:
            compare_verify(_np(v), ref["verify"], tally)
    tally.check_rate()


def test_stress_chained_rounds_match_oracle():
    """100 chained rounds of the stress workload (reduced vocabulary): x0 of round t+1
    is the last token round t emitted on the GPU, the RNG round index advances.  Every
    round is compared stage by stage; after a boundary case the oracle adopts the GPU's
    choice and the comparison goes on (no round or request is skipped)."""
    b = _b()
    wg, wn = _gpu_workload("stress", V=1032, rank=64, d=64)
    rd = b.Round(wg)
    x0_g = wg["x0"].clone()
    tally = Tally()
    R = wn["R"]
    for t in range(100):
        x0_h = x0_g.cpu().numpy()
        d, s, v = rd.run(rnd=t, x0=x0_g)
        torch.cuda.synchronize()
        gv = _np(v)
        check_round_stagewise(wg, wn, _np(d), _np(s), gv, t, x0_h, tally)
        last = gv["tokens"][np.arange(R), gv["n_out"] - 1]
        x0_g = torch.from_numpy(last.astype(np.int32)).cuda()
    assert tally.draws >= 100 * R * wn["gamma"]
    tally.check_rate()


@pytest.mark.parametrize("R,V,rank", [(5, 2056, 64), (32, 4104, 256), (64, 1032, 128), (100, 2056, 192),
                                      (200, 1160, 256), (513, 1032, 64)])
def test_draft_bias_dominant(R, V, rank):
    """Large low-rank factors (bias comparable to U), bf16: the tensor-core contraction
    decides the tokens, so any layout/descriptor error shows as token mismatches.
    Covers request blocks of 32/64/128 rows, several blocks, ragged R and V."""
    import torch
    b = _b()
    gamma, d = 3, 16
    g = torch.Generator().manual_seed(R * 7 + V)
    U = torch.randn((R, gamma, V), generator=g) * 1.0
    W1 = (torch.randn((V, rank), generator=g) * 0.35).to(torch.bfloat16)
    W2 = (torch.randn((rank, V), generator=g) * 0.35).to(torch.bfloat16)
    h = torch.randn((R, gamma, d), generator=g)
    cw = torch.randn(d + rank, generator=g) * 0.1
    x0 = torch.randint(0, V, (R,), generator=g, dtype=torch.int32)
    ids = torch.arange(R, dtype=torch.int64) * 3 + 1
    ct = torch.ones(gamma)
    gd = b.markov_draft(U.cuda(), W1.cuda(), W2.cuda(), h.cuda(), cw.cuda(), 0.0, 1.0, ct.cuda(), 1.0, x0.cuda(),
                        ids.cuda(), 5, 9)
    torch.cuda.synchronize()
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    od = oracle.markov_draft(U.numpy(), bits(W1), bits(W2), h.numpy(), cw.numpy(), 0.0, 1.0, ct.numpy(), 1.0,
                             x0.numpy(), ids.numpy(), 5, 9)
    tally = Tally()
    compare_draft(_np(gd), od, 2e-3, tally)
    # verification of the oracle's drafts: the residual recomputes the same bias rows
    target = torch.cat([U, U[:, -1:]], 1) + torch.randn((R, gamma + 1, V), generator=g) * 0.8
    ell = torch.randint(0, gamma + 1, (R,), generator=g, dtype=torch.int32)
    logq = od["logq"].astype(np.float32)
    lse = od["lse"].astype(np.float32)
    ov = oracle.verify(target.numpy(), U.numpy(), bits(W1), bits(W2), x0.numpy(), od["x"], logq, lse, ell.numpy(),
                       1.0, ids.numpy(), 5, 9)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    gv = b.verify(target.cuda(), U.cuda(), W1.cuda(), W2.cuda(), x0.cuda(), t(od["x"]), t(logq), t(lse), ell.cuda(),
                  1.0, ids.cuda(), 5, 9)
    torch.cuda.synchronize()
    compare_verify(_np(gv), ov, tally)
    assert (ov["corr_kind"] == 1).sum() >= min(R, 3)  # residual draws were exercised
    tally.check_rate()


def test_edge_cases():
    """Single request, gamma = 1, V not a multiple of 4/8 (scalar tails), zero-length and
    full-length verify, T != 1."""
    b = _b()
    rng = np.random.default_rng(3)
    for (R, gamma, V, rank, d, T) in ((1, 1, 5, 3, 1, 1.0), (3, 2, 37, 5, 0, 0.7), (2, 3, 1027, 64, 8, 1.3)):
        U = rng.normal(0, 1.5, (R, gamma, V)).astype(np.float32)
        target = np.concatenate([U, U[:, -1:]], 1) + rng.normal(0, 0.7, (R, gamma + 1, V)).astype(np.float32)
        target = target.astype(np.float32)
        W1 = rng.normal(0, 0.3, (V, rank)).astype(np.float32)
        W2 = rng.normal(0, 0.3, (rank, V)).astype(np.float32)
        h = rng.normal(0, 1, (R, gamma, max(d, 1))).astype(np.float32)[:, :, :d]
        cw = rng.normal(0, 0.5, d + rank).astype(np.float32)
        x0 = rng.integers(0, V, R).astype(np.int32)
        ids = (np.arange(R) * 7919 + 5).astype(np.int64)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        gd = b.markov_draft(t(U), t(W1), t(W2), t(h) if d > 0 else None, t(cw), 0.1, 1.2, t(np.ones(gamma, np.float32)),
                            T, t(x0), t(ids), 77, 4)
        od = oracle.markov_draft(U, W1, W2, h if d > 0 else np.zeros((R, gamma, 0), np.float32), cw, np.float32(0.1),
                                 np.float32(1.2), np.ones(gamma), T, x0, ids, 77, 4)
        tally = Tally()
        compare_draft(_np(gd), od, 1e-5, tally)
        for ell in (np.zeros(R, np.int32), np.full(R, gamma, np.int32)):
            ov = oracle.verify(target, U, W1, W2, x0, od["x"], od["logq"].astype(np.float32),
                               od["lse"].astype(np.float32), ell, T, ids, 77, 4)
            gv = b.verify(t(target), t(U), t(W1), t(W2), t(x0), t(od["x"]), t(od["logq"].astype(np.float32)),
                          t(od["lse"].astype(np.float32)), t(ell), T, t(ids), 77, 4)
            compare_verify(_np(gv), ov, tally)
        tally.check_rate()


def test_bad_device_inputs_reported_not_faulted():
    """An out-of-range anchor token or verify length is clamped in-kernel (every access
    stays in bounds) and reported through the workspace status word."""
    b = _b()
    wg, wn = _gpu_workload("tiny")
    x0 = wg["x0"].clone()
    x0[1] = wn["V"] + 5
    ws = b.workspace(b.draft_workspace_size(wn["R"], wn["gamma"], wn["V"], wn["rank"], wn["d"], torch.float32),
                     x0.device)
    b.markov_draft(wg["U"], wg["W1"], wg["W2"], wg["h"], wg["conf_w"], 0.0, 1.0, wg["conf_temp"], 1.0, x0,
                   wg["req_id"], 0, 0, ws=ws)
    assert b.device_status(ws, reset=True) == 1
    assert b.device_status(ws) == 0


def test_out_of_range_confidences_reported_not_faulted():
    """The scheduler's chains are sorted because c <= 1; a confidence outside [0,1] (or
    NaN) is reported and clamped, and the verify lengths stay valid."""
    b = _b()
    R, gamma = 16, 5
    conf = torch.rand((R, gamma), device="cuda", dtype=torch.float32)
    conf[3, 1] = 1.5
    conf[7, 0] = float("nan")
    conf[9, 4] = -0.25
    sps = torch.from_numpy(1000.0 / (1.0 + np.arange(R * (gamma + 1) + 1) / 64.0)).cuda()
    ws = b.workspace(b.schedule_workspace_size(R, gamma), conf.device)
    for mode in (0, 1, 2):
        out = b.schedule(conf, sps, mode, conf if mode == 2 else None, 0, ws=ws)
        torch.cuda.synchronize()
        assert b.device_status(ws, reset=True) == 1, mode
        ell = out["ell"].cpu().numpy()
        assert ((ell >= 0) & (ell <= gamma)).all()
        assert int(out["B"].item()) == R + int(ell.sum())


@pytest.mark.parametrize("R,gamma", [(1, 8), (3, 64), (5, 3), (100, 7), (513, 15), (700, 11), (8192, 1)])
def test_schedule_ragged_shapes_match_oracle(R, gamma):
    """Request counts that are not powers of two (partial merge lists), the largest
    gamma, and the largest candidate set; confidences with exact ties (1.0 and repeated
    values) so that the depth/request tie-break decides part of the order."""
    b = _b()
    rng = np.random.default_rng(R * 131 + gamma)
    conf = rng.choice(np.array([1.0, 0.999, 0.9, 0.5], np.float32), size=(R, gamma)).astype(np.float32)
    mix = rng.uniform(0.05, 1.0, (R, gamma)).astype(np.float32)
    conf = np.where(rng.uniform(size=(R, gamma)) < 0.5, conf, mix).astype(np.float32)
    hist = rng.uniform(0.0, 1.0, (R, gamma)).astype(np.float32)
    B = np.arange(R * (gamma + 1) + 1, dtype=np.float64)
    tally = Tally()
    for sps in (1000.0 / (1.0 + B / 64.0), np.where(B <= 2 * R, 1000.0, 1000.0 * 2 * R / np.maximum(B, 1.0))):
        sps = np.ascontiguousarray(sps)
        for mode in (wl.EARLY_STOP, wl.FULL_SEARCH, wl.CAPACITY_K):
            ref = oracle.schedule(conf, sps, mode, hist if mode == wl.CAPACITY_K else None)
            g = b.schedule(torch.from_numpy(conf).cuda(), torch.from_numpy(sps).cuda(), mode,
                           torch.from_numpy(hist).cuda() if mode == wl.CAPACITY_K else None)
            torch.cuda.synchronize()
            g = _np(g)
            compare_schedule(dict(ell=g["ell"], B=g["B"][0], tau=g["tau"][0]), ref, tally)
    tally.check_rate()


@pytest.mark.parametrize("R,gamma", [(1, 1), (4, 4), (32, 7), (513, 15), (8192, 1)])
def test_schedule_threshold_matches_oracle(R, gamma):
    """Fixed confidence cutoff: verify lengths and B bit-exact, tau within the fp64
    summation-order tolerance; cutoffs at, between and beyond the confidence values."""
    b = _b()
    rng = np.random.default_rng(R + 7 * gamma)
    conf = rng.choice(np.array([1.0, 0.75, 0.5, 0.25], np.float32), size=(R, gamma)).astype(np.float32)
    conf = np.where(rng.uniform(size=(R, gamma)) < 0.5, conf, rng.uniform(0, 1, (R, gamma))).astype(np.float32)
    conf[0, 0] = np.float32(np.nan) if R > 1 else conf[0, 0]
    for th in (0.0, 0.25, 0.5, 0.6, 0.75, 1.0, 1.5):
        ref = oracle.schedule_threshold(conf, th)
        g = _np(b.schedule_threshold(torch.from_numpy(conf).cuda(), th))
        torch.cuda.synchronize()
        assert np.array_equal(g["ell"], ref["ell"]), th
        assert int(g["B"][0]) == ref["B"], th
        assert abs(g["tau"][0] - ref["tau"]) <= 1e-12 * ref["tau"], th
