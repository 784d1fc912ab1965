"""Failure detection on the GPU without a fault: a bounded device wait that runs out.

The library is built a second time, for this test only, with a short wait limit
(DSPARK_TEST_WAIT_LIMIT, 2e6 cycles, about 1 ms) and a stall switch: a draft call whose
round index is 0x5EED has its U producer issue no copies, so each draft step's epilogue
waits on a shared-memory slot that nothing fills.  The wait gives up, records
DSPARK_TIMEOUT in the workspace's status word, lets the copies and MMAs already in
flight land, releases its tensor memory and returns.  The host reads status 5 through
dspark_workspace_status, and the next call on the same workspace (another round index)
runs normally and gives exactly the shipped library's results.  Nothing traps, faults or
hangs: every wait in the kernel is bounded.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from speculative_decoding_draft_03_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STALL_ROUND = 0x5EED


@pytest.fixture(scope="module")
def shortwait_lib():
    from speculative_decoding_draft_03_gb300 import build as bld
    path = bld.build(extra_flags=("-DDSPARK_TEST_WAIT_LIMIT=2000000ll",),
                     build_dir=os.path.join(ROOT, "tests", "_build", "shortwait"))
    lib = ctypes.CDLL(path)
    P, i32, u64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
    lib.dspark_markov_draft.argtypes = ([i32] * 8 + [P] * 4 + [P, f32, f32, P, f32, P, P, u64, u64] + [P] * 4
                                        + [P, sz, P])
    lib.dspark_markov_draft.restype = i32
    lib.dspark_workspace_status.argtypes = [P, i32, P, P]
    lib.dspark_workspace_status.restype = i32
    return lib


def _draft(lib, w, ws, out, rnd):
    from speculative_decoding_draft_03_gb300 import binding as b
    p = b._p
    st = lib.dspark_markov_draft(w["R"], w["gamma"], w["V"], w["rank"], w["d"], b._DT[w["U"].dtype],
                                 b._DT[w["W1"].dtype], b._DT[w["h"].dtype], p(w["U"]), p(w["W1"]), p(w["W2"]),
                                 p(w["h"]), p(w["conf_w"]), float(w["conf_b"]), float(w["conf_logit_scale"]),
                                 p(w["conf_temp"]), float(w["temperature"]), p(w["x0"]), p(w["req_id"]),
                                 int(w["seed"]), int(rnd), p(out["x"]), p(out["logq"]), p(out["lse"]),
                                 p(out["conf"]), p(ws), ws.numel(), b._stream())
    assert st == 0


def _status(lib, ws, reset):
    from speculative_decoding_draft_03_gb300 import binding as b
    val = ctypes.c_int(0)
    assert lib.dspark_workspace_status(b._p(ws), int(reset), ctypes.byref(val), b._stream()) == 0
    return int(val.value)


@pytest.mark.parametrize("name,over", [("qwen3-8b", dict(R=5, gamma=3, V=2056, d=64)),
                                       ("deepseek-v4", dict(R=200, gamma=2, V=4104, d=64))])
def test_bounded_wait_gives_up_and_reports_timeout(shortwait_lib, name, over):
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make(name, device="cuda", **over)
    R, gamma = w["R"], w["gamma"]
    dev = w["U"].device
    ws = b.workspace(b.draft_workspace_size(R, gamma, w["V"], w["rank"], w["d"], w["W1"].dtype), dev)
    mk = lambda: dict(x=torch.empty((R, gamma), dtype=torch.int32, device=dev),
                      logq=torch.empty((R, gamma), device=dev), lse=torch.empty((R, gamma), device=dev),
                      conf=torch.empty((R, gamma), device=dev))
    out = mk()
    _draft(shortwait_lib, w, ws, out, STALL_ROUND)
    torch.cuda.synchronize()  # the kernels returned: no hang, no fault
    assert _status(shortwait_lib, ws, reset=True) == 5  # DSPARK_TIMEOUT
    assert _status(shortwait_lib, ws, reset=False) == 0
    # the next call on the same workspace runs normally: the shipped library's results
    _draft(shortwait_lib, w, ws, out, 3)
    ref = b.markov_draft(w["U"], w["W1"], w["W2"], w["h"], w["conf_w"], w["conf_b"], w["conf_logit_scale"],
                         w["conf_temp"], w["temperature"], w["x0"], w["req_id"], w["seed"], 3, out=mk())
    torch.cuda.synchronize()
    assert _status(shortwait_lib, ws, reset=False) == 0
    for k in ("x", "logq", "lse", "conf"):
        assert torch.equal(out[k], ref[k]), k
    assert int(out["x"].min()) >= 0 and int(out["x"].max()) < w["V"]
