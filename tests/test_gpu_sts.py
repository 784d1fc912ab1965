"""dspark_sts_fit against the fp64 oracle.

The fit is a sequence of argmins over the temperature grid.  Each position is compared
given the GPU's own frozen temperatures for the earlier positions: the oracle evaluates
the ECE of every candidate in binary64, and the GPU's choice must reach the oracle's
minimum within a tolerance that covers samples whose fp32 prediction falls on the other
side of a bin edge (a few samples out of N); its reported ECE must equal the oracle's
ECE at the chosen temperature within the same tolerance.  Shapes cover several sample
chunks with a ragged tail, one bin, a single sample and position, a grid with unusable
candidates, and a closed-form case.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_03_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _fit(z, L, grid, M):
    from speculative_decoding_draft_03_gb300 import binding as b
    out = b.sts_fit(torch.as_tensor(z).cuda(), torch.as_tensor(L).cuda(), torch.as_tensor(grid).cuda(), M)
    torch.cuda.synchronize()
    return out["T"].cpu().numpy().astype(np.float64), out["ece"].cpu().numpy().astype(np.float64)


def _check(z, L, grid, M, T, ece):
    N, gamma = z.shape
    tol = 4.0 / N + 1e-6
    grid64 = grid.astype(np.float64)
    same = 0
    for k in range(1, gamma + 1):
        e_all = np.array([oracle.sts_ece(z, L, T[:k - 1], k, g, M) for g in grid64])
        valid = grid64 > 0
        e_all[~valid] = np.inf
        g_gpu = int(np.argmin(np.abs(grid64 - T[k - 1])))
        assert grid64[g_gpu] == T[k - 1]
        assert e_all[g_gpu] <= e_all.min() + tol, (k, e_all[g_gpu], e_all.min())
        assert abs(ece[k - 1] - e_all[g_gpu]) <= tol, (k, ece[k - 1], e_all[g_gpu])
        same += int(g_gpu == int(np.argmin(e_all)))
    return same


@pytest.mark.parametrize("N,T,M", [(20_000, (1.5, 0.7, 2.0, 1.0), 15),   # 5 chunks, ragged tail
                                   (4096, (0.5, 3.0), 10),                # exactly one chunk
                                   (9000, (1.2,), 1)])                    # one bin
def test_sts_fit_matches_oracle(N, T, M):
    d = wl.sts_heldout(N, len(T), T, seed=5)
    z, L = d["z"].numpy(), d["acc_len"].numpy()
    grid = wl.sts_grid(96)
    Tg, eg = _fit(z, L, grid, M)
    same = _check(z, L, grid, M, Tg, eg)
    assert same >= len(T) - 1  # at most one position decided by a near tie
    if M > 1:
        assert (np.abs(np.log(Tg) - np.log(np.asarray(T))) < 0.25).all(), Tg


def test_sts_fit_edges():
    # a single sample and position; unusable grid points are skipped
    z = np.array([[0.7]], np.float32)
    L = np.array([1], np.int32)
    grid = np.array([-1.0, 0.0, 0.5, 2.0, np.inf], np.float32)
    from speculative_decoding_draft_03_gb300 import binding as b
    ws = b.workspace(b.sts_fit_workspace_size(1, 1, len(grid), 4), "cuda")
    out = b.sts_fit(torch.as_tensor(z).cuda(), torch.as_tensor(L).cuda(), torch.as_tensor(grid).cuda(), 4, ws=ws)
    torch.cuda.synchronize()
    # p = sigmoid(0.7/T) is larger for the smaller T: the gap 1 - p is smallest at T = 0.5
    assert out["T"].item() == 0.5
    assert abs(out["ece"].item() - (1.0 - 1.0 / (1.0 + np.exp(-1.4)))) < 1e-6
    assert b.device_status(ws) == 1  # the non-positive / non-finite candidates were reported


def test_sts_fit_zero_logits_closed_form():
    N, gamma = 1000, 2
    z = np.zeros((N, gamma), np.float32)
    L = np.zeros(N, np.int32)
    L[:300] = 2
    L[300:500] = 1
    Tg, eg = _fit(z, L, np.array([0.5, 1.0, 2.0, 4.0], np.float32), 10)
    np.testing.assert_array_equal(Tg, [0.5, 0.5])
    np.testing.assert_allclose(eg, [0.0, 0.05], atol=1e-6)


@pytest.mark.slow
def test_sts_fit_full_size_local_optimality():
    # the configuration the benchmark times (131072 samples, 7 positions, 256 candidates):
    # at every position the GPU's temperature is at least as good as its grid neighbours
    # (given the GPU's earlier temperatures) and its reported ECE is the oracle's there
    N, gamma = 131072, 7
    T_true = [1.0 + 0.5 * ((k % 3) - 1) for k in range(gamma)]
    d = wl.sts_heldout(N, gamma, T_true, seed=0)
    z, L = d["z"].numpy(), d["acc_len"].numpy()
    grid = wl.sts_grid(256)
    Tg, eg = _fit(z, L, grid, 15)
    tol = 4.0 / N + 1e-6
    g64 = grid.astype(np.float64)
    for k in range(1, gamma + 1):
        gi = int(np.argmin(np.abs(g64 - Tg[k - 1])))
        e = oracle.sts_ece(z, L, Tg[:k - 1], k, g64[gi], 15)
        for nb in (gi - 1, gi + 1):
            if 0 <= nb < len(g64):
                assert e <= oracle.sts_ece(z, L, Tg[:k - 1], k, g64[nb], 15) + tol, (k, nb)
        assert abs(eg[k - 1] - e) <= tol, (k, eg[k - 1], e)


def test_sts_fit_single_candidate():
    d = wl.sts_heldout(3000, 2, (1.0, 2.0), seed=2)
    z, L = d["z"].numpy(), d["acc_len"].numpy()
    grid = np.array([1.7], np.float32)
    Tg, eg = _fit(z, L, grid, 12)
    np.testing.assert_array_equal(Tg, [grid[0], grid[0]])
    _check(z, L, grid, 12, Tg, eg)
