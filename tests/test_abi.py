"""The C-ABI library: it loads, exports exactly the symbols include/dspark.h declares,
and its host-side validation rejects bad arguments before anything is launched (these
calls never reach the GPU, so they run on CPU-only machines)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"DSPARK_API\s+[\w\s\*]*?\b(dspark_\w+)\s*\(", txt)))


@pytest.fixture(scope="module")
def b():
    from speculative_decoding_draft_03_gb300 import build
    build.build()
    from speculative_decoding_draft_03_gb300 import binding
    return binding


def test_exports_match_header(b):
    declared = _declared()
    assert len(declared) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", b._build.LIB], capture_output=True, text=True).stdout
    exported = sorted(set(m for m in re.findall(r"\bT\s+(\w+)", out)))
    assert exported == declared
    for name in declared:
        assert hasattr(b.lib, name)


def test_status_strings(b):
    for code, name in enumerate(["DSPARK_OK", "DSPARK_INVALID_ARG", "DSPARK_UNSUPPORTED_SHAPE",
                                 "DSPARK_WORKSPACE_TOO_SMALL", "DSPARK_CUDA_ERROR", "DSPARK_TIMEOUT"]):
        assert b.lib.dspark_status_string(code).decode() == name


def _fake(n=1):
    # distinct non-null, 256-aligned host-side stand-ins: validation never dereferences them
    return [ctypes.c_void_p(0x10000 + 0x1000 * i) for i in range(n)]


def _draft_call(b, **kw):
    args = dict(R=4, gamma=4, V=1024, rank=32, d=64, du=0, dw=0, dh=0, T=1.0, ws_bytes=1 << 30)
    args.update(kw)
    P = _fake(13)
    for k in kw.get("null", []):
        P[k] = None
    for k in kw.get("misalign", []):
        P[k] = ctypes.c_void_p(P[k].value + 8)
    return b.lib.dspark_markov_draft(args["R"], args["gamma"], args["V"], args["rank"], args["d"], args["du"],
                                     args["dw"], args["dh"], P[0], P[1], P[2], P[3], P[4], 0.0, 1.0, P[5],
                                     args["T"], P[6], P[7], 0, 0, P[8], P[9], P[10], P[11], P[12],
                                     args["ws_bytes"], None)


def test_draft_validation(b):
    assert _draft_call(b, R=0) == 1
    assert _draft_call(b, gamma=0) == 1
    assert _draft_call(b, rank=-1) == 1
    assert _draft_call(b, gamma=65) == 2
    assert _draft_call(b, du=7) == 1
    assert _draft_call(b, T=0.0) == 1
    assert _draft_call(b, T=float("nan")) == 1
    for k in (0, 1, 2, 4, 5, 6, 7, 8, 9, 10, 11, 12):
        assert _draft_call(b, null=[k]) == 1, k
    assert _draft_call(b, ws_bytes=16) == 3
    assert "workspace" in b.lib.dspark_last_error_message().decode()
    for k in (0, 1, 2, 3):  # U, W1, W2, h: 16-byte vector loads and TMA
        assert _draft_call(b, misalign=[k]) == 1, k
        assert "16-byte" in b.lib.dspark_last_error_message().decode()


def test_schedule_validation(b):
    P = _fake(6)
    L = b.lib.dspark_schedule
    assert L(0, 4, P[0], P[1], 100, 0, None, 0, P[2], P[3], P[4], P[5], 256, None) == 1
    assert L(4, 4, P[0], P[1], 100, 9, None, 0, P[2], P[3], P[4], P[5], 256, None) == 1
    assert L(4, 4, P[0], P[1], 10, 0, None, 0, P[2], P[3], P[4], P[5], 256, None) == 1  # sps too short
    assert L(4, 4, P[0], P[1], 100, 2, None, 0, P[2], P[3], P[4], P[5], 256, None) == 1  # capacity needs hist
    assert L(1024, 16, P[0], P[1], 1 << 20, 0, None, 0, P[2], P[3], P[4], P[5], 256, None) == 2
    assert L(4, 4, P[0], P[1], 100, 0, None, 0, P[2], P[3], P[4], P[5], 8, None) == 3
    assert L(4, 4, None, P[1], 100, 0, None, 0, P[2], P[3], P[4], P[5], 256, None) == 1


def test_verify_validation(b):
    P = _fake(17)
    L = b.lib.dspark_verify

    def call(**kw):
        a = dict(R=4, g=4, V=1024, rank=32, dt=0, T=1.0, ws=1 << 30)
        a.update(kw)
        p = list(P)
        for k in kw.get("null", []):
            p[k] = None
        for k in kw.get("misalign", []):
            p[k] = ctypes.c_void_p(p[k].value + 4)
        return L(a["R"], a["g"], a["V"], a["rank"], a["dt"], 0, 0, p[0], p[1], p[2], p[3], p[4], p[5], p[6],
                 p[7], p[8], a["T"], p[9], 0, 0, p[10], p[11], p[12], p[13], a["ws"], None)

    assert call(R=0) == 1
    assert call(g=100) == 2
    assert call(dt=3) == 1
    assert call(T=-1.0) == 1
    for k in range(14):
        assert call(null=[k]) == 1, k
    assert call(ws=100) == 3
    for k in (0, 1, 2, 3):  # target, U, W1, W2
        assert call(misalign=[k]) == 1, k
        assert "16-byte" in b.lib.dspark_last_error_message().decode()


def test_verify_overlap_validation(b):
    import torch
    P = _fake(18)
    L = b.lib.dspark_verify_overlap
    need = b.verify_overlap_workspace_size(4, 4, 1024, 32, torch.float32)

    def call(**kw):
        a = dict(R=4, g=4, V=1024, rank=32, dt=0, T=1.0, ws=need)
        a.update(kw)
        p = list(P)
        for k in kw.get("null", []):
            p[k] = None
        return L(a["R"], a["g"], a["V"], a["rank"], a["dt"], 0, 0, p[0], p[1], p[2], p[3], p[4], p[5], p[6],
                 p[7], p[8], a["T"], p[9], 0, 0, p[10], p[11], p[12], p[13], p[14], a["ws"], None)

    assert call(R=0) == 1
    assert call(g=100) == 2
    assert call(T=0.0) == 1
    for k in range(15):  # every pointer, overlap_out and the workspace included
        assert call(null=[k]) == 1, k
    # the fused call needs the verify workspace plus the overlap pass's pieces
    assert need > b.verify_workspace_size(4, 4, 1024, 32, torch.float32)
    assert call(ws=b.verify_workspace_size(4, 4, 1024, 32, torch.float32)) == 3
    assert call(ws=need - 1) == 3
    assert b.verify_overlap_workspace_size(0, 4, 1024, 32, torch.float32) == 0


def test_overlap_workspaces_stay_linear_in_rows(b):
    # the compact tensor-core pass keeps one partial per SM per row only while its row
    # blocks fit on the SMs; larger batches take the flattened path, whose partials do not
    # grow with the grid (no quadratic growth in R * gamma)
    import torch
    bf = torch.bfloat16
    for fn in (b.acceptance_overlap_workspace_size, b.verify_overlap_workspace_size):
        small = fn(4096, 16, 151936, 256, bf)
        big = fn(65536, 16, 151936, 256, bf)
        assert 0 < small < big < 20 * small, (fn.__name__, small, big)


def test_workspace_sizes_grow_with_shape(b):
    import torch
    s1 = b.draft_workspace_size(4, 4, 1024, 32, 64, torch.float32)
    s2 = b.draft_workspace_size(32, 7, 151936, 256, 4096, torch.bfloat16)
    assert 256 < s1 < s2
    assert b.verify_workspace_size(4, 4, 1024, 32, torch.float32) > 256
    assert b.schedule_workspace_size(512, 15) >= 256


def test_verify_ragged_validation(b):
    P = _fake(18)
    L = b.lib.dspark_verify_ragged

    def call(**kw):
        a = dict(R=4, g=4, V=1024, rank=32, nrows=10, ws=1 << 30)
        a.update(kw)
        p = list(P)
        for k in kw.get("null", []):
            p[k] = None
        for k in kw.get("misalign", []):
            p[k] = ctypes.c_void_p(p[k].value + 4)
        return L(a["R"], a["g"], a["V"], a["rank"], 0, 0, 0, p[0], a["nrows"], p[1], p[2], p[3], p[4], p[5], p[6],
                 p[7], p[8], p[9], 1.0, p[10], 0, 0, p[11], p[12], p[13], p[14], a["ws"], None)

    assert call(nrows=0) == 1
    assert call(null=[1]) == 1  # row offsets
    assert "target_row_offset" in b.lib.dspark_last_error_message().decode()
    assert call(null=[0]) == 1
    assert call(misalign=[0]) == 1
    assert call(R=0) == 1
    assert call(ws=100) == 3


def test_schedule_threshold_validation(b):
    P = _fake(5)
    L = b.lib.dspark_schedule_threshold
    call = lambda R=4, g=4, th=0.5, ws=1 << 20, null=(): L(R, g, *([None if k in null else P[k] for k in range(1)]),
                                                           th, *([None if k in null else P[k] for k in range(1, 5)]),
                                                           ws, None)
    assert call(R=0) == 1
    assert call(g=65) == 2
    assert call(th=float("nan")) == 1
    for k in range(5):
        assert call(null=(k,)) == 1, k
    assert call(ws=16) == 3


def test_acceptance_overlap_validation(b):
    P = _fake(10)
    L = b.lib.dspark_acceptance_overlap

    def call(**kw):
        a = dict(R=4, g=4, V=1024, rank=32, dt=0, T=1.0, ws=1 << 30)
        a.update(kw)
        p = list(P)
        for k in kw.get("null", []):
            p[k] = None
        for k in kw.get("misalign", []):
            p[k] = ctypes.c_void_p(p[k].value + 4)
        return L(a["R"], a["g"], a["V"], a["rank"], a["dt"], 0, 0, p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7],
                 a["T"], p[8], p[9], a["ws"], None)

    assert call(R=0) == 1
    assert call(g=100) == 2
    assert call(dt=3) == 1
    assert call(T=0.0) == 1
    for k in (0, 1, 2, 3, 4, 5, 6, 8, 9):  # every pointer but ell (optional)
        assert call(null=[k]) == 1, k
    for k in (0, 1, 2, 3):
        assert call(misalign=[k]) == 1, k
    assert call(ws=100) == 3
    assert call(null=[7], ws=100) == 3  # a missing ell is allowed: the next check fails
    assert b.acceptance_overlap_workspace_size(4, 4, 1024, 32, __import__("torch").float32) > 256
    assert b.acceptance_overlap_workspace_size(0, 4, 1024, 32, __import__("torch").float32) == 0


def test_rnn_draft_validation(b):
    P = _fake(22)
    L = b.lib.dspark_rnn_draft

    def call(**kw):
        a = dict(R=4, g=4, V=1024, ns=32, ne=32, d=64, du=0, T=1.0, ws=1 << 30)
        a.update(kw)
        p = list(P)
        for k in kw.get("null", []):
            p[k] = None
        for k in kw.get("misalign", []):
            p[k] = ctypes.c_void_p(p[k].value + 4)
        return L(a["R"], a["g"], a["V"], a["ns"], a["ne"], a["d"], a["du"], 0, 0, p[0], p[1], p[2], p[3], p[4], p[5],
                 p[6], p[7], 0.0, 1.0, p[8], a["T"], p[9], p[10], 0, 0, p[11], p[12], p[13], p[14], p[15], p[16],
                 a["ws"], None)

    assert call(R=0) == 1
    assert call(ne=-1) == 1
    assert call(g=100) == 2
    assert call(ns=48) == 2  # not a multiple of 32
    assert call(ns=288) == 2
    assert call(ne=4096) == 2
    assert call(du=5) == 1
    assert call(T=0.0) == 1
    # U, E, Wse, Wh, bgc, Wo, h, conf_w, conf_temp, x0, req_id, outputs, state, workspace
    for k in range(17):
        assert call(null=[k]) == 1, k
    assert call(null=[1], ne=0, ws=100) == 3  # no embedding: E may be missing
    assert call(null=[3, 6], d=0, ws=100) == 3  # no hidden state: Wh and h may be missing
    for k in (0, 3, 5, 6):  # U, Wh, Wo, h
        assert call(misalign=[k]) == 1, k
    assert call(ws=100) == 3
    import torch
    assert b.rnn_draft_workspace_size(4, 4, 1024, 32, 64, torch.float32) > b.draft_workspace_size(
        4, 4, 1024, 32, 64, torch.float32)


def test_verify_rnn_validation(b):
    P = _fake(17)
    L = b.lib.dspark_verify_rnn

    def call(**kw):
        p = list(P)
        for k in kw.get("null", []):
            p[k] = None
        return L(4, 4, 1024, 32, 0, 0, 0, p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8], 1.0, p[9], 0, 0,
                 p[10], p[11], p[12], p[13], kw.get("ws", 1 << 30), None)

    for k in range(14):
        assert call(null=[k]) == 1, k
    assert "state" in (call(null=[2]) and b.lib.dspark_last_error_message().decode())
    assert call(ws=100) == 3


def test_sts_fit_validation(b):
    P = _fake(6)
    L = b.lib.dspark_sts_fit

    def call(N=100, g=4, G=8, M=15, ws=1 << 30, null=()):
        p = [None if k in null else P[k] for k in range(6)]
        return L(N, g, p[0], p[1], p[2], G, M, p[3], p[4], p[5], ws, None)

    assert call(N=0) == 1
    assert call(G=0) == 1
    assert call(M=0) == 1
    assert call(g=65) == 2
    assert call(M=17) == 2
    assert call(G=70000) == 2
    for k in range(6):
        assert call(null=(k,)) == 1, k
    assert call(ws=100) == 3
    assert b.sts_fit_workspace_size(100, 4, 8, 15) > 256


def test_header_is_plain_c(tmp_path):
    # the boundary carries no C++ or CUDA types: the header compiles as C99 on its own
    src = tmp_path / "use.c"
    src.write_text('#include "dspark.h"\nint main(void) { return DSPARK_OK + (int)sizeof(dspark_status); }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-fsyntax-only",
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
