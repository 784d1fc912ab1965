"""fp64 CPU oracle of the DSpark per-round hot path (draft -> schedule -> verify).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this package.
The product library never loads it; the two share no code.

The arithmetic lives in ``dspark_oracle.c`` (plain C, binary64, OpenMP over
independent requests).  This module only compiles it with gcc, loads it with ctypes
and marshals numpy arrays.  Function docstrings name the page and section each step
follows; the C file states the steps themselves.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

F32, BF16 = 0, 1
EARLY_STOP, FULL_SEARCH, CAPACITY_K, FIXED = 0, 1, 2, 3
STREAM_DRAFT, STREAM_ACCEPT, STREAM_CORRECT = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no FMA contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wno-unknown-pragmas", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, u32, u64, f64 = ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
            lib.orc_philox4x32_10.argtypes = [P, P, P]
            lib.orc_draw_bits.argtypes = [u64, u64, u64, u32, u32, u32, u32]
            lib.orc_draw_bits.restype = u32
            lib.orc_uniform.argtypes = [u32]
            lib.orc_uniform.restype = f64
            lib.orc_gumbel.argtypes = [f64]
            lib.orc_gumbel.restype = f64
            lib.orc_markov_draft.argtypes = [i32] * 8 + [P] * 4 + [P, f64, f64, P, f64, P, P, u64, u64] + [P] * 6 + [i32]
            lib.orc_draft_distribution.argtypes = [i32, i32, i32, i32, P, P, P, i32, f64, P]
            lib.orc_schedule.argtypes = [i32, i32, P, P, i32, i32, P, i32, P, P, P, P]
            lib.orc_schedule_path.argtypes = [i32, i32, P, P, P, P, P, P]
            lib.orc_schedule_many.argtypes = [i32, i32, i32, P, P, i32, i32, P, i32, P]
            lib.orc_schedule_many.restype = ctypes.c_int
            lib.orc_schedule_threshold.argtypes = [i32, i32, P, f64, P, P, P]
            lib.orc_schedule_threshold.restype = ctypes.c_int
            lib.orc_verify.argtypes = ([i32] * 7 + [P] * 4 + [P, P, P, P, P, f64, P, u64, u64]
                                       + [P] * 3 + [P] * 4 + [P, i32])
            lib.orc_rnn_cell.argtypes = [i32] * 5 + [P, i32] + [P] * 5 + [ctypes.c_size_t, P]
            lib.orc_rnn_cell.restype = ctypes.c_int
            lib.orc_draft_row.argtypes = [i32] * 4 + [P, P, P, f64, u64, u64, u64, u32] + [P] * 5
            lib.orc_draft_row.restype = ctypes.c_int
            lib.orc_rnn_draft.argtypes = ([i32] * 9 + [P] * 7 + [P, f64, f64, P, f64, P, P, u64, u64]
                                          + [P] * 7 + [i32])
            lib.orc_rnn_draft.restype = ctypes.c_int
            lib.orc_rnn_confidence.argtypes = [i32] * 5 + [P, P, P, f64, f64, P, P]
            lib.orc_rnn_confidence.restype = ctypes.c_int
            lib.orc_sts_ece.argtypes = [i32, i32, P, P, P, i32, f64, i32]
            lib.orc_sts_ece.restype = f64
            lib.orc_sts_fit.argtypes = [i32, i32, P, P, P, i32, i32, P, P]
            lib.orc_sts_fit.restype = ctypes.c_int
            lib.orc_max_threads.restype = i32
            lib.orc_acceptance_overlap.argtypes = [i32] * 7 + [P] * 7 + [f64, P, i32]
            lib.orc_acceptance_overlap.restype = ctypes.c_int
            for name in ("orc_markov_draft", "orc_draft_distribution", "orc_schedule",
                         "orc_schedule_path", "orc_verify", "orc_philox4x32_10"):
                getattr(lib, name).restype = ctypes.c_int if name != "orc_philox4x32_10" else None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dtype_code(a):
    if a.dtype == np.float32:
        return F32, a
    if a.dtype == np.uint16:  # raw bf16 bit patterns
        return BF16, a
    raise TypeError(f"oracle takes float32 or raw-bf16 (uint16) arrays, got {a.dtype}")


def max_threads() -> int:
    return int(_load().orc_max_threads())


# ---------------------------------------------------------------------------
# Counter-based random numbers (Philox4x32-10, Salmon et al. SC'11)
# ---------------------------------------------------------------------------
def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: 4 counter words, 2 key words -> 4 output words."""
    lib = _load()
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib.orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def draw_bits(seed, req_id, rnd, stream, position, chunk, lane) -> int:
    return int(_load().orc_draw_bits(seed, req_id, rnd, stream, position, chunk, lane))


def uniform(bits) -> float:
    return float(_load().orc_uniform(bits))


def gumbel(u) -> float:
    return float(_load().orc_gumbel(u))


# ---------------------------------------------------------------------------
# Stage 1: Markov-head draft + confidence head
# ---------------------------------------------------------------------------
def markov_draft(U, W1, W2, h, conf_w, conf_b, conf_logit_scale, conf_temp, temperature,
                 x0, req_id, seed, rnd, nthreads=0):
    """Draft gamma tokens per request (numb3r33 blog "Markov sequential head"; DSpark 精读 §2, §4).

    U [R,gamma,V], W1 [V,rank], W2 [rank,V], h [R,gamma,d]: float32 or raw bf16 (uint16).
    Returns dict: x [R,gamma] int32, logq, lse, conf (float64), runner_up, margin.
    """
    lib = _load()
    du, U = _dtype_code(np.ascontiguousarray(U))
    dw, W1 = _dtype_code(np.ascontiguousarray(W1))
    dw2, W2 = _dtype_code(np.ascontiguousarray(W2))
    dh, h = _dtype_code(np.ascontiguousarray(h))
    assert dw == dw2
    R, gamma, V = U.shape
    rank = W1.shape[1]
    d = h.shape[2]
    conf_w = _c(conf_w, np.float32)
    conf_temp = _c(conf_temp, np.float32)
    x0 = _c(x0, np.int32)
    req_id = _c(req_id, np.int64)
    out = dict(x=np.zeros((R, gamma), np.int32), logq=np.zeros((R, gamma)), lse=np.zeros((R, gamma)),
               conf=np.zeros((R, gamma)), runner_up=np.zeros((R, gamma), np.int32),
               margin=np.zeros((R, gamma)))
    rc = lib.orc_markov_draft(R, gamma, V, rank, d, du, dw, dh, _ptr(U), _ptr(W1), _ptr(W2), _ptr(h),
                              _ptr(conf_w), float(conf_b), float(conf_logit_scale), _ptr(conf_temp),
                              float(temperature), _ptr(x0), _ptr(req_id), int(seed), int(rnd),
                              _ptr(out["x"]), _ptr(out["logq"]), _ptr(out["lse"]), _ptr(out["conf"]),
                              _ptr(out["runner_up"]), _ptr(out["margin"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle markov_draft rejected its arguments")
    return out


def draft_distribution(U_row, W1, W2, x_prev, temperature):
    """Full q_k(.|x_prev) = softmax((U_k + W1[x_prev] W2)/T) over the vocabulary (test helper)."""
    lib = _load()
    du, U_row = _dtype_code(np.ascontiguousarray(U_row))
    dw, W1 = _dtype_code(np.ascontiguousarray(W1))
    _, W2 = _dtype_code(np.ascontiguousarray(W2))
    V = U_row.shape[-1]
    q = np.zeros(V)
    lib.orc_draft_distribution(V, W1.shape[1], du, dw, _ptr(U_row), _ptr(W1), _ptr(W2), int(x_prev),
                               float(temperature), _ptr(q))
    return q


# ---------------------------------------------------------------------------
# Stage 2: confidence scheduler
# ---------------------------------------------------------------------------
def schedule(conf, sps, mode, conf_hist=None, fixed_len=0):
    """Per-request verify lengths maximising tau*SPS(B) (DSpark 精读 §4; vllmbangkok §4.2.2).

    conf [R,gamma] float32; sps float64 indexed by B. Returns dict ell, B, tau, gap, tie.
    """
    lib = _load()
    conf = _c(conf, np.float32)
    R, gamma = conf.shape
    sps = _c(sps, np.float64)
    hist = None if conf_hist is None else _c(conf_hist, np.float32)
    ell = np.zeros(R, np.int32)
    B = np.zeros(1, np.int32)
    tau = np.zeros(1)
    diag = np.zeros(2)
    rc = lib.orc_schedule(R, gamma, _ptr(conf), _ptr(sps), len(sps), int(mode), _ptr(hist),
                          int(fixed_len), _ptr(ell), _ptr(B), _ptr(tau), _ptr(diag))
    if rc != 0:
        raise ValueError("oracle schedule rejected its arguments")
    return dict(ell=ell, B=int(B[0]), tau=float(tau[0]), gap=float(diag[0]), tie=float(diag[1]))


def schedule_threshold(conf, threshold):
    """Verify lengths from a fixed confidence cutoff: each request keeps its leading drafts
    with c >= threshold (vllmbangkok "Verify smarter, not longer").  Returns ell, B, tau."""
    lib = _load()
    conf = _c(conf, np.float32)
    R, gamma = conf.shape
    ell = np.zeros(R, np.int32)
    B = np.zeros(1, np.int32)
    tau = np.zeros(1)
    rc = lib.orc_schedule_threshold(R, gamma, _ptr(conf), ctypes.c_double(float(threshold)), _ptr(ell), _ptr(B),
                                    _ptr(tau))
    if rc != 0:
        raise ValueError("oracle schedule_threshold rejected its arguments")
    return dict(ell=ell, B=int(B[0]), tau=float(tau[0]))


def schedule_many(conf, sps, mode, conf_hist=None, fixed_len=0):
    """Independent scheduler problems: conf [nbatch,R,gamma] -> ell [nbatch,R]."""
    lib = _load()
    conf = _c(conf, np.float32)
    nb, R, gamma = conf.shape
    sps = _c(sps, np.float64)
    hist = None if conf_hist is None else _c(conf_hist, np.float32)
    ell = np.zeros((nb, R), np.int32)
    rc = lib.orc_schedule_many(nb, R, gamma, _ptr(conf), _ptr(sps), len(sps), int(mode), _ptr(hist),
                               int(fixed_len), _ptr(ell))
    if rc != 0:
        raise ValueError("oracle schedule rejected its arguments")
    return ell


def schedule_path(conf, sps):
    """Sorted admission path: a_(n), its request and depth, and Theta(n) for n=0..N."""
    lib = _load()
    conf = _c(conf, np.float32)
    R, gamma = conf.shape
    sps = _c(sps, np.float64)
    N = R * gamma
    a = np.zeros(N)
    req = np.zeros(N, np.int32)
    dep = np.zeros(N, np.int32)
    theta = np.zeros(N + 1)
    lib.orc_schedule_path(R, gamma, _ptr(conf), _ptr(sps), _ptr(a), _ptr(req), _ptr(dep), _ptr(theta))
    return dict(a=a, req=req, depth=dep, theta=theta)


# ---------------------------------------------------------------------------
# Stage 3: exact verification
# ---------------------------------------------------------------------------
def verify(target, U, W1, W2, x0, x, logq, lse_q, ell, temperature, req_id, seed, rnd, nthreads=0, state=None):
    """min(1,p/q) acceptance, (p-q)+ residual, bonus token (numb3r33 blog "One-token exactness").

    target [R,gamma+1,V]; x [R,gamma]; logq, lse_q [R,gamma] (float64 or float32); ell [R].
    state [R,gamma,rank] (recurrent head): the residual's factor rows (W1 is then unused).
    Returns dict n_acc, tokens [R,gamma+1], n_out, acc_margin, corr_margin, corr_rho, corr_kind.
    """
    lib = _load()
    dt, target = _dtype_code(np.ascontiguousarray(target))
    du, U = _dtype_code(np.ascontiguousarray(U))
    dw1, W1 = _dtype_code(np.ascontiguousarray(W1))
    dw, W2 = _dtype_code(np.ascontiguousarray(W2))
    if state is None and dw1 != dw:
        raise TypeError("W1 and W2 must have the same storage type")
    R, g1, V = target.shape
    gamma = g1 - 1
    x0 = _c(x0, np.int32)
    x = _c(x, np.int32)
    logq = _c(logq, np.float64)
    lse_q = _c(lse_q, np.float64)
    ell = _c(ell, np.int32)
    req_id = _c(req_id, np.int64)
    st = None if state is None else _c(state, np.float64)
    rank = W1.shape[1] if st is None else st.shape[2]
    out = dict(n_acc=np.zeros(R, np.int32), tokens=np.zeros((R, gamma + 1), np.int32),
               n_out=np.zeros(R, np.int32), acc_margin=np.zeros((R, gamma)),
               corr_margin=np.zeros(R), corr_rho=np.zeros((R, 2)), corr_kind=np.zeros(R, np.int32))
    rc = lib.orc_verify(R, gamma, V, rank, dt, du, dw, _ptr(target), _ptr(U), _ptr(W1), _ptr(W2),
                        _ptr(x0), _ptr(x), _ptr(logq), _ptr(lse_q), _ptr(ell), float(temperature),
                        _ptr(req_id), int(seed), int(rnd), _ptr(out["n_acc"]), _ptr(out["tokens"]),
                        _ptr(out["n_out"]), _ptr(out["acc_margin"]), _ptr(out["corr_margin"]),
                        _ptr(out["corr_rho"]), _ptr(out["corr_kind"]), _ptr(st), int(nthreads))
    if rc != 0:
        raise ValueError("oracle verify rejected its arguments")
    return out


# ---------------------------------------------------------------------------
# Stage 1, recurrent head (numb3r33 blog "RNN sequential head"; DSpark 精读 §2)
# ---------------------------------------------------------------------------
def rnn_cell(s_prev, x_prev, E, Wse, Wh, bgc, h_row):
    """One gated state update s = (1-g) s_prev + g tanh(.) on [s_prev; E[x_prev]; h_row],
    rounded to the weights' storage type.  s_prev float64 [ns] (stored values)."""
    lib = _load()
    dw, E = _dtype_code(np.ascontiguousarray(E))
    _, Wse = _dtype_code(np.ascontiguousarray(Wse))
    _, Wh = _dtype_code(np.ascontiguousarray(Wh))
    dh, h_row = _dtype_code(np.ascontiguousarray(h_row))
    ns = Wse.shape[1] // 2
    ne = E.shape[1]
    d = h_row.shape[-1]
    s_prev = _c(s_prev, np.float64)
    bgc = _c(bgc, np.float32)
    out = np.zeros(ns)
    rc = lib.orc_rnn_cell(ns, ne, d, dw, dh, _ptr(s_prev), int(x_prev), _ptr(E), _ptr(Wse), _ptr(Wh), _ptr(bgc),
                          _ptr(h_row), 0, _ptr(out))
    if rc != 0:
        raise ValueError("oracle rnn_cell rejected its arguments")
    return out


def draft_row(U_row, arow, W2, temperature, seed, req_id, rnd, position):
    """One draft position given its factor row: (x, lse, logq, runner_up, margin)."""
    lib = _load()
    du, U_row = _dtype_code(np.ascontiguousarray(U_row))
    dw, W2 = _dtype_code(np.ascontiguousarray(W2))
    arow = _c(arow, np.float64)
    x = np.zeros(1, np.int32)
    ru = np.zeros(1, np.int32)
    lse, logq, mg = np.zeros(1), np.zeros(1), np.zeros(1)
    lib.orc_draft_row(U_row.shape[-1], arow.shape[0], du, dw, _ptr(U_row), _ptr(arow), _ptr(W2), float(temperature),
                      int(seed), int(req_id), int(rnd), int(position), _ptr(x), _ptr(lse), _ptr(logq), _ptr(ru),
                      _ptr(mg))
    return dict(x=int(x[0]), lse=float(lse[0]), logq=float(logq[0]), runner_up=int(ru[0]), margin=float(mg[0]))


def rnn_confidence(h, state, conf_w, conf_b, conf_logit_scale, conf_temp):
    """c[r,k] = sigmoid(kappa (w_h . h[r,k] + w_s . state[r,k] + b) / T_k) for given states."""
    lib = _load()
    dh, h = _dtype_code(np.ascontiguousarray(h))
    state = _c(state, np.float64)
    R, gamma, d = h.shape
    ns = state.shape[2]
    out = np.zeros((R, gamma))
    lib.orc_rnn_confidence(R, gamma, d, ns, dh, _ptr(h), _ptr(state), _ptr(_c(conf_w, np.float32)), float(conf_b),
                           float(conf_logit_scale), _ptr(_c(conf_temp, np.float32)), _ptr(out))
    return out


def rnn_draft(U, E, Wse, Wh, bgc, Wo, h, conf_w, conf_b, conf_logit_scale, conf_temp, temperature, x0, req_id,
              seed, rnd, nthreads=0):
    """Draft loop with the recurrent head.  U [R,gamma,V]; E [V,ne]; Wse [ns+ne,2ns];
    Wh [d,2ns]; bgc [2ns]; Wo [ns,V]; h [R,gamma,d]; conf_w [d+ns].
    Returns dict x, logq, lse, conf, state [R,gamma,ns], runner_up, margin."""
    lib = _load()
    du, U = _dtype_code(np.ascontiguousarray(U))
    dw, E = _dtype_code(np.ascontiguousarray(E))
    _, Wse = _dtype_code(np.ascontiguousarray(Wse))
    _, Wh = _dtype_code(np.ascontiguousarray(Wh))
    _, Wo = _dtype_code(np.ascontiguousarray(Wo))
    dh, h = _dtype_code(np.ascontiguousarray(h))
    R, gamma, V = U.shape
    ns = Wse.shape[1] // 2
    ne = E.shape[1]
    d = h.shape[2]
    bgc = _c(bgc, np.float32)
    conf_w = _c(conf_w, np.float32)
    conf_temp = _c(conf_temp, np.float32)
    x0 = _c(x0, np.int32)
    req_id = _c(req_id, np.int64)
    out = dict(x=np.zeros((R, gamma), np.int32), logq=np.zeros((R, gamma)), lse=np.zeros((R, gamma)),
               conf=np.zeros((R, gamma)), state=np.zeros((R, gamma, ns)), runner_up=np.zeros((R, gamma), np.int32),
               margin=np.zeros((R, gamma)))
    rc = lib.orc_rnn_draft(R, gamma, V, ns, ne, d, du, dw, dh, _ptr(U), _ptr(E), _ptr(Wse), _ptr(Wh), _ptr(bgc),
                           _ptr(Wo), _ptr(h), _ptr(conf_w), float(conf_b), float(conf_logit_scale), _ptr(conf_temp),
                           float(temperature), _ptr(x0), _ptr(req_id), int(seed), int(rnd), _ptr(out["x"]),
                           _ptr(out["logq"]), _ptr(out["lse"]), _ptr(out["conf"]), _ptr(out["state"]),
                           _ptr(out["runner_up"]), _ptr(out["margin"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rnn_draft rejected its arguments")
    return out


def acceptance_overlap(target, U, W1, W2, x0, x, ell=None, temperature=1.0, nthreads=0):
    """Expected acceptance of each drafted position, c*_j = sum_v min(q_j(v), p_j(v))
    (numb3r33 blog, "Total variation label").

    target [R,gamma+1,V]; U [R,gamma,V]; x [R,gamma]; ell [R] or None (every position).
    Returns float64 [R,gamma], NaN at positions past ell[r].
    """
    lib = _load()
    dt, target = _dtype_code(np.ascontiguousarray(target))
    du, U = _dtype_code(np.ascontiguousarray(U))
    dw, W1 = _dtype_code(np.ascontiguousarray(W1))
    _, W2 = _dtype_code(np.ascontiguousarray(W2))
    R, g1, V = target.shape
    gamma = g1 - 1
    x0 = _c(x0, np.int32)
    x = _c(x, np.int32)
    ell_c = None if ell is None else _c(ell, np.int32)
    out = np.zeros((R, gamma))
    rc = lib.orc_acceptance_overlap(R, gamma, V, W1.shape[1], dt, du, dw, _ptr(target), _ptr(U), _ptr(W1),
                                    _ptr(W2), _ptr(x0), _ptr(x), _ptr(ell_c), float(temperature), _ptr(out),
                                    int(nthreads))
    if rc != 0:
        raise ValueError("oracle acceptance_overlap rejected its arguments")
    return out


# ---------------------------------------------------------------------------
# Sequential temperature scaling (numb3r33 blog "Sequential temperature scaling";
# mkdocs.reaper.mx "3 · DSpark" §3.2)
# ---------------------------------------------------------------------------
def sts_ece(z, acc_len, T_prev, k, T, M):
    """ECE of the cumulative survival at position k (1-based) for temperature T, with
    the temperatures of positions 1..k-1 frozen at T_prev."""
    z = _c(z, np.float32)
    N, gamma = z.shape
    acc = _c(acc_len, np.int32)
    tp = _c(np.asarray(T_prev, np.float64).reshape(-1) if len(T_prev) else np.zeros(1), np.float64)
    return float(_load().orc_sts_ece(N, gamma, _ptr(z), _ptr(acc), _ptr(tp), int(k), float(T), int(M)))


def sts_fit(z, acc_len, grid, M):
    """Per-position temperatures fitted left to right on held-out (z, L) pairs.
    z [N,gamma] confidence logits; acc_len [N] accepted drafts; grid [G] candidates.
    Returns (T [gamma], ece [gamma])."""
    z = _c(z, np.float32)
    N, gamma = z.shape
    acc = _c(acc_len, np.int32)
    grid = _c(grid, np.float64)
    T = np.zeros(gamma)
    ece = np.zeros(gamma)
    rc = _load().orc_sts_fit(N, gamma, _ptr(z), _ptr(acc), _ptr(grid), len(grid), int(M), _ptr(T), _ptr(ece))
    if rc != 0:
        raise ValueError("oracle sts_fit rejected its arguments")
    return T, ece


def run_round(inp, rnd=0, x0=None, conf_hist=None, nthreads=0):
    """One full round: draft -> schedule (on float32 confidences, the type the stages
    exchange) -> verify (on float32 logq / lse, likewise).  ``inp`` is a workload dict."""
    x0 = inp["x0"] if x0 is None else x0
    rnn = inp.get("head") == "rnn"
    if rnn:
        d = rnn_draft(inp["U"], inp["E"], inp["Wse"], inp["Wh"], inp["bgc"], inp["Wo"], inp["h"], inp["conf_w"],
                      inp["conf_b"], inp["conf_logit_scale"], inp["conf_temp"], inp["temperature"], x0,
                      inp["req_id"], inp["seed"], rnd, nthreads)
    else:
        d = markov_draft(inp["U"], inp["W1"], inp["W2"], inp["h"], inp["conf_w"], inp["conf_b"],
                         inp["conf_logit_scale"], inp["conf_temp"], inp["temperature"], x0,
                         inp["req_id"], inp["seed"], rnd, nthreads)
    conf32 = d["conf"].astype(np.float32)
    hist = inp.get("conf_hist") if conf_hist is None else conf_hist
    s = schedule(conf32, inp["sps"], inp["mode"], hist, inp.get("fixed_len", 0))
    W1 = np.zeros((1, 1), inp["Wo"].dtype) if rnn else inp["W1"]
    W2 = inp["Wo"] if rnn else inp["W2"]
    v = verify(inp["target"], inp["U"], W1, W2, x0, d["x"],
               d["logq"].astype(np.float32), d["lse"].astype(np.float32), s["ell"],
               inp["temperature"], inp["req_id"], inp["seed"], rnd, nthreads, state=d["state"] if rnn else None)
    return dict(draft=d, sched=s, verify=v)
