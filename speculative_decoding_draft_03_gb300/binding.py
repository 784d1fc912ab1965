"""Thin ctypes binding of ``libdspark.so`` (argument marshalling only).

Every step of the path runs in the library's CUDA kernels; this module checks tensor
placement/dtypes, passes ``data_ptr()``s and the current CUDA stream, and owns the
caller-side buffers (outputs and workspaces) through PyTorch.  If the library is
missing this module raises at import: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

F32, BF16 = 0, 1
EARLY_STOP, FULL_SEARCH, CAPACITY_K, FIXED = 0, 1, 2, 3
_DT = {torch.float32: F32, torch.bfloat16: BF16}


class DSparkError(RuntimeError):
    pass


def _load_library():
    path = _build.LIB
    if not os.path.exists(path):
        raise DSparkError(f"libdspark.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, i32, u64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
    lib.dspark_status_string.restype = ctypes.c_char_p
    lib.dspark_status_string.argtypes = [i32]
    lib.dspark_last_error_message.restype = ctypes.c_char_p
    lib.dspark_workspace_status.argtypes = [P, i32, P, P]
    lib.dspark_markov_draft_workspace_size.restype = sz
    lib.dspark_markov_draft_workspace_size.argtypes = [i32] * 5 + [i32]
    lib.dspark_markov_draft.argtypes = ([i32] * 8 + [P] * 4 + [P, f32, f32, P, f32, P, P, u64, u64]
                                        + [P] * 4 + [P, sz, P])
    lib.dspark_schedule_workspace_size.restype = sz
    lib.dspark_schedule_workspace_size.argtypes = [i32, i32]
    lib.dspark_schedule.argtypes = [i32, i32, P, P, i32, i32, P, i32, P, P, P, P, sz, P]
    lib.dspark_schedule_threshold.argtypes = [i32, i32, P, ctypes.c_double, P, P, P, P, sz, P]
    lib.dspark_schedule_threshold.restype = i32
    lib.dspark_verify_workspace_size.restype = sz
    lib.dspark_verify_workspace_size.argtypes = [i32] * 5
    lib.dspark_verify.argtypes = ([i32] * 7 + [P] * 4 + [P] * 5 + [f32, P, u64, u64] + [P] * 3 + [P, sz, P])
    lib.dspark_set_profile_events.argtypes = [P, i32]
    lib.dspark_set_profile_events.restype = None
    lib.dspark_set_verify_profile_events.argtypes = [P, i32]
    lib.dspark_set_verify_profile_events.restype = None
    lib.dspark_verify_ragged.argtypes = ([i32] * 7 + [P, i32, P] + [P] * 3 + [P] * 5 + [f32, P, u64, u64] + [P] * 3
                                         + [P, sz, P])
    lib.dspark_verify_ragged.restype = i32
    lib.dspark_verify_static.argtypes = ([i32] * 7 + [P] * 4 + [P] * 5 + [f32, P, u64, u64] + [P] * 3 + [P])
    lib.dspark_verify_static.restype = i32
    lib.dspark_verify_static_status.argtypes = [i32, P, P]
    lib.dspark_verify_static_status.restype = i32
    lib.dspark_verify_overlap_workspace_size.restype = sz
    lib.dspark_verify_overlap_workspace_size.argtypes = [i32] * 5
    lib.dspark_verify_overlap.argtypes = ([i32] * 7 + [P] * 4 + [P] * 5 + [f32, P, u64, u64] + [P] * 4
                                          + [P, sz, P])
    lib.dspark_verify_overlap.restype = i32
    lib.dspark_acceptance_overlap_workspace_size.restype = sz
    lib.dspark_acceptance_overlap_workspace_size.argtypes = [i32] * 5
    lib.dspark_acceptance_overlap.argtypes = [i32] * 7 + [P] * 4 + [P] * 4 + [f32, P, P, sz, P]
    lib.dspark_acceptance_overlap.restype = i32
    lib.dspark_rnn_draft_workspace_size.restype = sz
    lib.dspark_rnn_draft_workspace_size.argtypes = [i32] * 6
    lib.dspark_rnn_draft.argtypes = ([i32] * 9 + [P] * 7 + [P, f32, f32, P, f32, P, P, u64, u64] + [P] * 5
                                     + [P, sz, P])
    lib.dspark_rnn_draft.restype = i32
    lib.dspark_verify_rnn.argtypes = ([i32] * 7 + [P] * 4 + [P] * 5 + [f32, P, u64, u64] + [P] * 3 + [P, sz, P])
    lib.dspark_verify_rnn.restype = i32
    lib.dspark_sts_fit_workspace_size.restype = sz
    lib.dspark_sts_fit_workspace_size.argtypes = [i32] * 4
    lib.dspark_sts_fit.argtypes = [i32, i32, P, P, P, i32, i32, P, P, P, sz, P]
    lib.dspark_sts_fit.restype = i32
    for fn in ("dspark_markov_draft", "dspark_schedule", "dspark_verify", "dspark_workspace_status"):
        getattr(lib, fn).restype = i32
    return lib


lib = _load_library()


def _check(status: int, what: str):
    if status != 0:
        name = lib.dspark_status_string(status).decode()
        msg = lib.dspark_last_error_message().decode()
        raise DSparkError(f"{what}: {name}: {msg}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise DSparkError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise DSparkError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise DSparkError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _dt(t, name):
    if t.dtype not in _DT:
        raise DSparkError(f"{name} must be float32 or bfloat16, got {t.dtype}")
    return _DT[t.dtype]


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A caller-owned, 256-byte aligned device workspace whose status word starts at 0."""
    ws = torch.zeros(max(256, int(nbytes)) + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + max(256, int(nbytes))]


def draft_workspace_size(R, gamma, V, rank, d, w_dtype) -> int:
    return int(lib.dspark_markov_draft_workspace_size(R, gamma, V, rank, d, _DT[w_dtype]))


def schedule_workspace_size(R, gamma) -> int:
    return int(lib.dspark_schedule_workspace_size(R, gamma))


def verify_workspace_size(R, gamma, V, rank, w_dtype) -> int:
    return int(lib.dspark_verify_workspace_size(R, gamma, V, rank, _DT[w_dtype]))


def markov_draft(U, W1, W2, h, conf_w, conf_b, conf_logit_scale, conf_temp, temperature, x0, req_id,
                 seed, rnd, out=None, ws=None, stream=None):
    """Stage 1 (dspark_markov_draft).  Returns dict x, logq, lse, conf (device tensors)."""
    R, gamma, V = U.shape
    rank = W1.shape[1]
    d = h.shape[2] if h is not None else 0
    dev = U.device
    for t, n in ((U, "U"), (W1, "W1"), (W2, "W2")):
        _cuda(t, n)
    if h is not None:
        _cuda(h, "h")
    _cuda(conf_w, "conf_w", torch.float32)
    _cuda(conf_temp, "conf_temp", torch.float32)
    _cuda(x0, "x0", torch.int32)
    _cuda(req_id, "req_id", torch.int64)
    if W1.dtype != W2.dtype:
        raise DSparkError("W1 and W2 must share a dtype")
    if out is None:
        out = dict(x=torch.empty((R, gamma), dtype=torch.int32, device=dev),
                   logq=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   lse=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   conf=torch.empty((R, gamma), dtype=torch.float32, device=dev))
    if ws is None:
        ws = workspace(draft_workspace_size(R, gamma, V, rank, d, W1.dtype), dev)
    st = lib.dspark_markov_draft(R, gamma, V, rank, d, _dt(U, "U"), _dt(W1, "W1"),
                                 _dt(h, "h") if h is not None else F32,
                                 _p(U), _p(W1), _p(W2), _p(h), _p(conf_w), float(conf_b),
                                 float(conf_logit_scale), _p(conf_temp), float(temperature), _p(x0),
                                 _p(req_id), int(seed), int(rnd), _p(out["x"]), _p(out["logq"]),
                                 _p(out["lse"]), _p(out["conf"]), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dspark_markov_draft")
    return out


def schedule(conf, sps, mode, conf_hist=None, fixed_len=0, out=None, ws=None, stream=None):
    """Stage 2 (dspark_schedule).  Returns dict ell [R] int32, B [1] int32, tau [1] float64."""
    _cuda(conf, "conf", torch.float32)
    R, gamma = conf.shape
    dev = conf.device
    if sps is not None:
        _cuda(sps, "sps", torch.float64)
    if conf_hist is not None:
        _cuda(conf_hist, "conf_hist", torch.float32)
    if out is None:
        out = dict(ell=torch.empty(R, dtype=torch.int32, device=dev),
                   B=torch.empty(1, dtype=torch.int32, device=dev),
                   tau=torch.empty(1, dtype=torch.float64, device=dev))
    if ws is None:
        ws = workspace(schedule_workspace_size(R, gamma), dev)
    st = lib.dspark_schedule(R, gamma, _p(conf), _p(sps), 0 if sps is None else sps.numel(), int(mode),
                             _p(conf_hist), int(fixed_len), _p(out["ell"]), _p(out["B"]), _p(out["tau"]),
                             _p(ws), ws.numel(), _stream(stream))
    _check(st, "dspark_schedule")
    return out


def schedule_threshold(conf, threshold, out=None, ws=None, stream=None):
    """Stage 2 with a fixed confidence cutoff (dspark_schedule_threshold).  Returns dict
    ell [R] int32, B [1] int32, tau [1] float64."""
    _cuda(conf, "conf", torch.float32)
    R, gamma = conf.shape
    dev = conf.device
    if out is None:
        out = dict(ell=torch.empty(R, dtype=torch.int32, device=dev),
                   B=torch.empty(1, dtype=torch.int32, device=dev),
                   tau=torch.empty(1, dtype=torch.float64, device=dev))
    if ws is None:
        ws = workspace(schedule_workspace_size(R, gamma), dev)
    st = lib.dspark_schedule_threshold(R, gamma, _p(conf), float(threshold), _p(out["ell"]), _p(out["B"]),
                                       _p(out["tau"]), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dspark_schedule_threshold")
    return out


def verify(target, U, W1, W2, x0, x, logq, lse_q, ell, temperature, req_id, seed, rnd, out=None,
           ws=None, stream=None):
    """Stage 3 (dspark_verify).  Returns dict n_acc [R], tokens [R,gamma+1], n_out [R]."""
    R, g1, V = target.shape
    gamma = g1 - 1
    rank = W1.shape[1]
    dev = target.device
    for t, n in ((target, "target"), (U, "U"), (W1, "W1"), (W2, "W2")):
        _cuda(t, n)
    _cuda(x0, "x0", torch.int32)
    _cuda(x, "x", torch.int32)
    _cuda(logq, "logq", torch.float32)
    _cuda(lse_q, "lse_q", torch.float32)
    _cuda(ell, "ell", torch.int32)
    _cuda(req_id, "req_id", torch.int64)
    if out is None:
        out = dict(n_acc=torch.empty(R, dtype=torch.int32, device=dev),
                   tokens=torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty(R, dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(verify_workspace_size(R, gamma, V, rank, W1.dtype), dev)
    st = lib.dspark_verify(R, gamma, V, rank, _dt(target, "target"), _dt(U, "U"), _dt(W1, "W1"),
                           _p(target), _p(U), _p(W1), _p(W2), _p(x0), _p(x), _p(logq), _p(lse_q), _p(ell),
                           float(temperature), _p(req_id), int(seed), int(rnd), _p(out["n_acc"]),
                           _p(out["tokens"]), _p(out["n_out"]), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dspark_verify")
    return out


def verify_ragged(target_rows, row_offset, U, W1, W2, x0, x, logq, lse_q, ell, temperature, req_id, seed, rnd,
                  out=None, ws=None, stream=None):
    """Stage 3 on a flattened target (dspark_verify_ragged): target_rows [n_rows, V],
    request r's verify rows at row_offset[r] + t.  Returns dict n_acc, tokens, n_out."""
    n_rows, V = target_rows.shape
    R, gamma = x.shape
    rank = W1.shape[1]
    dev = target_rows.device
    for t, n in ((target_rows, "target_rows"), (U, "U"), (W1, "W1"), (W2, "W2")):
        _cuda(t, n)
    _cuda(row_offset, "row_offset", torch.int32)
    _cuda(x0, "x0", torch.int32)
    _cuda(x, "x", torch.int32)
    _cuda(logq, "logq", torch.float32)
    _cuda(lse_q, "lse_q", torch.float32)
    _cuda(ell, "ell", torch.int32)
    _cuda(req_id, "req_id", torch.int64)
    if out is None:
        out = dict(n_acc=torch.empty(R, dtype=torch.int32, device=dev),
                   tokens=torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty(R, dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(verify_workspace_size(R, gamma, V, rank, W1.dtype), dev)
    st = lib.dspark_verify_ragged(R, gamma, V, rank, _dt(target_rows, "target_rows"), _dt(U, "U"), _dt(W1, "W1"),
                                  _p(target_rows), int(n_rows), _p(row_offset), _p(U), _p(W1), _p(W2), _p(x0),
                                  _p(x), _p(logq), _p(lse_q), _p(ell), float(temperature), _p(req_id), int(seed),
                                  int(rnd), _p(out["n_acc"]), _p(out["tokens"]), _p(out["n_out"]), _p(ws),
                                  ws.numel(), _stream(stream))
    _check(st, "dspark_verify_ragged")
    return out


def verify_overlap_workspace_size(R, gamma, V, rank, w_dtype) -> int:
    return int(lib.dspark_verify_overlap_workspace_size(R, gamma, V, rank, _DT[w_dtype]))


def verify_overlap(target, U, W1, W2, x0, x, logq, lse_q, ell, temperature, req_id, seed, rnd, out=None,
                   ws=None, stream=None):
    """Stage 3 with the acceptance overlap fused in (dspark_verify_overlap).  Returns dict
    n_acc [R], tokens [R,gamma+1], n_out [R] and overlap [R,gamma] (NaN past ell[r])."""
    R, g1, V = target.shape
    gamma = g1 - 1
    rank = W1.shape[1]
    dev = target.device
    for t, n in ((target, "target"), (U, "U"), (W1, "W1"), (W2, "W2")):
        _cuda(t, n)
    _cuda(x0, "x0", torch.int32)
    _cuda(x, "x", torch.int32)
    _cuda(logq, "logq", torch.float32)
    _cuda(lse_q, "lse_q", torch.float32)
    _cuda(ell, "ell", torch.int32)
    _cuda(req_id, "req_id", torch.int64)
    if out is None:
        out = dict(n_acc=torch.empty(R, dtype=torch.int32, device=dev),
                   tokens=torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty(R, dtype=torch.int32, device=dev),
                   overlap=torch.empty((R, gamma), dtype=torch.float32, device=dev))
    if ws is None:
        ws = workspace(verify_overlap_workspace_size(R, gamma, V, rank, W1.dtype), dev)
    st = lib.dspark_verify_overlap(R, gamma, V, rank, _dt(target, "target"), _dt(U, "U"), _dt(W1, "W1"),
                                   _p(target), _p(U), _p(W1), _p(W2), _p(x0), _p(x), _p(logq), _p(lse_q), _p(ell),
                                   float(temperature), _p(req_id), int(seed), int(rnd), _p(out["n_acc"]),
                                   _p(out["tokens"]), _p(out["n_out"]), _p(out["overlap"]), _p(ws), ws.numel(),
                                   _stream(stream))
    _check(st, "dspark_verify_overlap")
    return out


def acceptance_overlap_workspace_size(R, gamma, V, rank, w_dtype) -> int:
    return int(lib.dspark_acceptance_overlap_workspace_size(R, gamma, V, rank, _DT[w_dtype]))


def acceptance_overlap(target, U, W1, W2, x0, x, lse_q, ell, temperature, out=None, ws=None, stream=None):
    """Expected acceptance c*[r,j] = sum_v min(q_j, p_j) of every drafted position
    (dspark_acceptance_overlap); ell None evaluates all positions.  Returns [R,gamma]
    float32, NaN past ell[r]."""
    R, g1, V = target.shape
    gamma = g1 - 1
    rank = W1.shape[1]
    dev = target.device
    for t, n in ((target, "target"), (U, "U"), (W1, "W1"), (W2, "W2")):
        _cuda(t, n)
    _cuda(x0, "x0", torch.int32)
    _cuda(x, "x", torch.int32)
    _cuda(lse_q, "lse_q", torch.float32)
    if ell is not None:
        _cuda(ell, "ell", torch.int32)
    if out is None:
        out = torch.empty((R, gamma), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(acceptance_overlap_workspace_size(R, gamma, V, rank, W1.dtype), dev)
    st = lib.dspark_acceptance_overlap(R, gamma, V, rank, _dt(target, "target"), _dt(U, "U"), _dt(W1, "W1"),
                                       _p(target), _p(U), _p(W1), _p(W2), _p(x0), _p(x), _p(lse_q), _p(ell),
                                       float(temperature), _p(out), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dspark_acceptance_overlap")
    return out


def rnn_draft_workspace_size(R, gamma, V, ns, d, w_dtype) -> int:
    return int(lib.dspark_rnn_draft_workspace_size(R, gamma, V, ns, d, _DT[w_dtype]))


def rnn_draft(U, E, Wse, Wh, bgc, Wo, h, conf_w, conf_b, conf_logit_scale, conf_temp, temperature, x0, req_id,
              seed, rnd, out=None, ws=None, stream=None):
    """Stage 1 with the recurrent head (dspark_rnn_draft).  Returns dict x, logq, lse, conf,
    state [R,gamma,ns]."""
    R, gamma, V = U.shape
    ns = Wo.shape[0]
    ne = E.shape[1] if E is not None else 0
    d = h.shape[2] if h is not None else 0
    dev = U.device
    for t, n in ((U, "U"), (Wse, "Wse"), (Wo, "Wo")):
        _cuda(t, n)
    if ne:
        _cuda(E, "E")
    if d:
        _cuda(Wh, "Wh")
        _cuda(h, "h")
    _cuda(bgc, "bgc", torch.float32)
    _cuda(conf_w, "conf_w", torch.float32)
    _cuda(conf_temp, "conf_temp", torch.float32)
    _cuda(x0, "x0", torch.int32)
    _cuda(req_id, "req_id", torch.int64)
    if out is None:
        out = dict(x=torch.empty((R, gamma), dtype=torch.int32, device=dev),
                   logq=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   lse=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   conf=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                   state=torch.empty((R, gamma, ns), dtype=Wo.dtype, device=dev))
    if ws is None:
        ws = workspace(rnn_draft_workspace_size(R, gamma, V, ns, d, Wo.dtype), dev)
    st = lib.dspark_rnn_draft(R, gamma, V, ns, ne, d, _dt(U, "U"), _dt(Wo, "Wo"), _dt(h, "h") if d else F32,
                              _p(U), _p(E) if ne else None, _p(Wse), _p(Wh) if d else None, _p(bgc), _p(Wo),
                              _p(h) if d else None, _p(conf_w), float(conf_b), float(conf_logit_scale),
                              _p(conf_temp), float(temperature), _p(x0), _p(req_id), int(seed), int(rnd),
                              _p(out["x"]), _p(out["logq"]), _p(out["lse"]), _p(out["conf"]), _p(out["state"]),
                              _p(ws), ws.numel(), _stream(stream))
    _check(st, "dspark_rnn_draft")
    return out


def verify_rnn(target, U, state, Wo, x0, x, logq, lse_q, ell, temperature, req_id, seed, rnd, out=None, ws=None,
               stream=None):
    """Stage 3 for a block drafted by the recurrent head (dspark_verify_rnn)."""
    R, g1, V = target.shape
    gamma = g1 - 1
    ns = Wo.shape[0]
    dev = target.device
    for t, n in ((target, "target"), (U, "U"), (state, "state"), (Wo, "Wo")):
        _cuda(t, n)
    _cuda(x0, "x0", torch.int32)
    _cuda(x, "x", torch.int32)
    _cuda(logq, "logq", torch.float32)
    _cuda(lse_q, "lse_q", torch.float32)
    _cuda(ell, "ell", torch.int32)
    _cuda(req_id, "req_id", torch.int64)
    if out is None:
        out = dict(n_acc=torch.empty(R, dtype=torch.int32, device=dev),
                   tokens=torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty(R, dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(verify_workspace_size(R, gamma, V, ns, Wo.dtype), dev)
    st = lib.dspark_verify_rnn(R, gamma, V, ns, _dt(target, "target"), _dt(U, "U"), _dt(Wo, "Wo"), _p(target),
                               _p(U), _p(state), _p(Wo), _p(x0), _p(x), _p(logq), _p(lse_q), _p(ell),
                               float(temperature), _p(req_id), int(seed), int(rnd), _p(out["n_acc"]),
                               _p(out["tokens"]), _p(out["n_out"]), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dspark_verify_rnn")
    return out


def sts_fit_workspace_size(N, gamma, G, M) -> int:
    return int(lib.dspark_sts_fit_workspace_size(N, gamma, G, M))


def sts_fit(z, acc_len, grid, M, out=None, ws=None, stream=None):
    """Per-position confidence temperatures fitted left to right on held-out samples
    (dspark_sts_fit).  z [N,gamma] fp32 logits, acc_len [N] int32, grid [G] fp32.
    Returns dict T [gamma], ece [gamma]."""
    N, gamma = z.shape
    G = grid.shape[0]
    _cuda(z, "z", torch.float32)
    _cuda(acc_len, "acc_len", torch.int32)
    _cuda(grid, "grid", torch.float32)
    dev = z.device
    if out is None:
        out = dict(T=torch.empty(gamma, dtype=torch.float32, device=dev),
                   ece=torch.empty(gamma, dtype=torch.float32, device=dev))
    if ws is None:
        ws = workspace(sts_fit_workspace_size(N, gamma, G, M), dev)
    st = lib.dspark_sts_fit(N, gamma, _p(z), _p(acc_len), _p(grid), G, int(M), _p(out["T"]), _p(out["ece"]), _p(ws),
                            ws.numel(), _stream(stream))
    _check(st, "dspark_sts_fit")
    return out


def verify_static(target, U, W1, W2, x0, x, logq, lse_q, ell, temperature, req_id, seed, rnd, out=None,
                  stream=None):
    """Stage 3 through dspark_verify_static: for callers that cannot allocate device
    memory (a pooled allocator they must not bypass, allocation-free serving loops); the
    scratch is the library's own static array, so concurrent calls on one device must
    be ordered by the caller."""
    R, g1, V = target.shape
    gamma = g1 - 1
    rank = W1.shape[1]
    dev = target.device
    for t, n in ((target, "target"), (U, "U"), (W1, "W1"), (W2, "W2")):
        _cuda(t, n)
    _cuda(x0, "x0", torch.int32)
    _cuda(x, "x", torch.int32)
    _cuda(logq, "logq", torch.float32)
    _cuda(lse_q, "lse_q", torch.float32)
    _cuda(ell, "ell", torch.int32)
    _cuda(req_id, "req_id", torch.int64)
    if out is None:
        out = dict(n_acc=torch.empty(R, dtype=torch.int32, device=dev),
                   tokens=torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty(R, dtype=torch.int32, device=dev))
    st = lib.dspark_verify_static(R, gamma, V, rank, _dt(target, "target"), _dt(U, "U"), _dt(W1, "W1"),
                                  _p(target), _p(U), _p(W1), _p(W2), _p(x0), _p(x), _p(logq), _p(lse_q), _p(ell),
                                  float(temperature), _p(req_id), int(seed), int(rnd), _p(out["n_acc"]),
                                  _p(out["tokens"]), _p(out["n_out"]), _stream(stream))
    _check(st, "dspark_verify_static")
    return out


def verify_static_status(reset=False, stream=None) -> int:
    """The device status word of dspark_verify_static's scratch on the current device: what
    the last call's kernels reported (0 OK, 1 bad device data, 5 a bounded wait gave up)."""
    val = ctypes.c_int(0)
    _check(lib.dspark_verify_static_status(int(reset), ctypes.byref(val), _stream(stream)),
           "dspark_verify_static_status")
    return int(val.value)


class StepTimer:
    """Times the draft stage's vocabulary-streaming step kernel (one launch per draft
    position) with CUDA events the library records around each launch."""

    def __init__(self, gamma: int):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * gamma)]
        for e in self.events:
            e.record()  # materialise the handles
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self.samples = []

    def __enter__(self):
        lib.dspark_set_profile_events(self._arr, len(self.events))
        return self

    def __exit__(self, *exc):
        lib.dspark_set_profile_events(None, 0)

    def collect(self):
        """After the stream has synchronised: append this round's per-launch times (ms)."""
        for k in range(len(self.events) // 2):
            self.samples.append(self.events[2 * k].elapsed_time(self.events[2 * k + 1]))


class VerifyTimer:
    """Times verification's two vocabulary-streaming kernels, the target-row statistics
    pass and the correction pass, with CUDA events the library records around them."""

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in self.events:
            e.record()
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in self.events])
        self.rows, self.correction = [], []

    def __enter__(self):
        lib.dspark_set_verify_profile_events(self._arr, 4)
        return self

    def __exit__(self, *exc):
        lib.dspark_set_verify_profile_events(None, 0)

    def collect(self):
        """After the stream has synchronised: append this round's two times (ms)."""
        self.rows.append(self.events[0].elapsed_time(self.events[1]))
        self.correction.append(self.events[2].elapsed_time(self.events[3]))


def device_status(ws, reset=False, stream=None) -> int:
    """The workspace's device status word (0 OK, 5 a bounded wait gave up, 1 bad device data)."""
    val = ctypes.c_int(0)
    _check(lib.dspark_workspace_status(_p(ws), int(reset), ctypes.byref(val), _stream(stream)),
           "dspark_workspace_status")
    return int(val.value)


class Round:
    """One DSpark round (draft -> schedule -> verify) over a fixed workload shape, with
    every output and workspace allocated once, so that repeated rounds (and CUDA-graph
    capture) launch kernels only."""

    def __init__(self, w: dict):
        self.w = w
        R, gamma, V, rank, d = w["R"], w["gamma"], w["V"], w["rank"], w["d"]
        dev = w["U"].device
        self.draft_out = dict(x=torch.empty((R, gamma), dtype=torch.int32, device=dev),
                              logq=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                              lse=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                              conf=torch.empty((R, gamma), dtype=torch.float32, device=dev))
        self.sched_out = dict(ell=torch.empty(R, dtype=torch.int32, device=dev),
                              B=torch.empty(1, dtype=torch.int32, device=dev),
                              tau=torch.empty(1, dtype=torch.float64, device=dev))
        self.verify_out = dict(n_acc=torch.empty(R, dtype=torch.int32, device=dev),
                               tokens=torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
                               n_out=torch.empty(R, dtype=torch.int32, device=dev))
        self.rnn = w.get("head") == "rnn"
        if self.rnn:
            self.draft_out["state"] = torch.empty((R, gamma, rank), dtype=w["Wo"].dtype, device=dev)
            self.ws_draft = workspace(rnn_draft_workspace_size(R, gamma, V, rank, d, w["Wo"].dtype), dev)
        else:
            self.ws_draft = workspace(draft_workspace_size(R, gamma, V, rank, d, w["W1"].dtype), dev)
        self.ws_sched = workspace(schedule_workspace_size(R, gamma), dev)
        wdt = w["Wo"].dtype if self.rnn else w["W1"].dtype
        self.ws_verify = workspace(verify_workspace_size(R, gamma, V, rank, wdt), dev)
        self.x0 = w["x0"].clone()

    def run(self, rnd=0, x0=None, stream=None):
        w = self.w
        x0 = self.x0 if x0 is None else x0
        if self.rnn:
            d = rnn_draft(w["U"], w["E"], w["Wse"], w["Wh"], w["bgc"], w["Wo"], w["h"], w["conf_w"], w["conf_b"],
                          w["conf_logit_scale"], w["conf_temp"], w["temperature"], x0, w["req_id"], w["seed"], rnd,
                          out=self.draft_out, ws=self.ws_draft, stream=stream)
        else:
            d = markov_draft(w["U"], w["W1"], w["W2"], w["h"], w["conf_w"], w["conf_b"], w["conf_logit_scale"],
                             w["conf_temp"], w["temperature"], x0, w["req_id"], w["seed"], rnd,
                             out=self.draft_out, ws=self.ws_draft, stream=stream)
        s = schedule(d["conf"], w["sps"], w["mode"], w.get("conf_hist"), w.get("fixed_len", 0),
                     out=self.sched_out, ws=self.ws_sched, stream=stream)
        if self.rnn:
            v = verify_rnn(w["target"], w["U"], d["state"], w["Wo"], x0, d["x"], d["logq"], d["lse"], s["ell"],
                           w["temperature"], w["req_id"], w["seed"], rnd, out=self.verify_out, ws=self.ws_verify,
                           stream=stream)
        else:
            v = verify(w["target"], w["U"], w["W1"], w["W2"], x0, d["x"], d["logq"], d["lse"], s["ell"],
                       w["temperature"], w["req_id"], w["seed"], rnd, out=self.verify_out, ws=self.ws_verify,
                       stream=stream)
        return d, s, v

    def capture(self, rnd=0, x0=None, timer=None):
        """Capture one round (round index ``rnd``) as a CUDA graph.  Replaying it launches
        the round's kernels with no host work; it writes the same output tensors as
        ``run``.  With ``timer`` (a StepTimer) the graph also records its step events."""
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=self.w["U"].device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=side):
            if timer is not None:
                with timer:
                    self.run(rnd, x0)
            else:
                self.run(rnd, x0)
        torch.cuda.current_stream().wait_stream(side)
        return g

    def status(self) -> int:
        codes = [device_status(ws) for ws in (self.ws_draft, self.ws_sched, self.ws_verify)]
        return max(codes)
