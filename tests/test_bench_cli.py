"""bench.py's command line and the pieces of its JSON line that need no GPU: the options
parse, every workload has a description, the stored ncu counters are used only when they
were taken on the current kernel sources, the per-round acceptance figures and the
byte counts of the verification kernels, and the draw-by-draw round comparison."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_help_lists_every_mode():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr
    for opt in ("--gpus", "--steps", "--warmup", "--impl", "--workload", "--head", "--diagnostic", "--no-others"):
        assert opt in r.stdout, opt
    for mode in ("overlap", "verify_overlap", "sts"):
        assert mode in r.stdout, mode


def test_defaults_are_the_headline_workload():
    import bench
    a = bench.parse([])
    assert a.workload == "stress" and a.gpus == 1 and a.warmup >= 3


def test_workload_descriptions_and_stored_counters(tmp_path):
    import bench
    from speculative_decoding_draft_03_gb300 import workloads as wl
    for name in wl.SHAPES:
        assert bench.WORKLOAD_DESC[name]
    t = bench.stored_traffic("draft_step", "qwen3-8b")
    # either the committed counters match the kernel source (then the DRAM bytes are about
    # the algorithmic 97.26 MB per launch), or the traffic is reported as unknown
    assert t is None or 90e6 < t < 110e6, t
    # a stale source hash hides the entry; a matching one exposes it
    src = ["bench.py"]
    p = tmp_path / "c.json"
    p.write_text(json.dumps({"k": {"w": {"sources": src, "source_sha": "0" * 16, "traffic_bytes_per_launch": 5}}}))
    assert bench.stored_traffic("k", "w", str(p)) is None
    p.write_text(json.dumps({"k": {"w": {"sources": src, "source_sha": bench.source_hash(src),
                                         "traffic_bytes_per_launch": 5}}}))
    assert bench.stored_traffic("k", "w", str(p)) == 5.0
    assert bench.stored_traffic("missing", "w", str(p)) is None


def test_acceptance_stats():
    import bench
    ell = [[2, 0, 3], [1, 1, 0]]
    acc = [[2, 0, 1], [0, 1, 0]]
    s = bench.acceptance_stats(3, ell, acc)
    assert s["rounds"] == 2
    assert s["sum_ell_per_round"] == (5 + 2) / 2
    assert s["sum_n_acc_per_round"] == (3 + 1) / 2
    assert s["verify_batch_B_per_round"] == (8 + 5) / 2
    # depth 1 verified by 4 requests (2, 3 | 1, 1), accepted by 3
    assert s["verified_at_depth"][0] == 4 and s["conditional_acceptance_by_depth"][0] == 0.75
    # depth 2: verified with depth 1 accepted: (2, 3) -> accepted by the first only
    assert s["verified_at_depth"][1] == 2 and s["conditional_acceptance_by_depth"][1] == 0.5
    assert s["verified_at_depth"][2] == 0 and s["conditional_acceptance_by_depth"][2] is None


def test_verify_byte_counts():
    import torch
    import bench
    w = dict(R=3, V=1000, rank=64, U=torch.zeros(1, dtype=torch.float32), target=torch.zeros(1, dtype=torch.bfloat16),
             W2=torch.zeros(1, dtype=torch.bfloat16))
    assert bench.verify_rows_bytes(w, [2, 0, 3]) == (3 + 1 + 4) * 1000 * 2
    # one rejection (request 2: 1 accepted of 3)
    assert bench.correction_bytes(w, [2, 0, 3], [2, 0, 1]) == 1000 * (4 + 2) + 64 * 1000 * 2


def test_compare_round_counts_boundaries():
    import bench
    R, g = 2, 3
    ref = {"draft": {"x": np.array([[1, 2, 3], [4, 5, 6]]), "margin": np.full((R, g), 1.0),
                     "runner_up": np.zeros((R, g), int)},
           "sched": {"ell": np.array([2, 1]), "gap": 1.0, "tie": 1.0},
           "verify": {"n_acc": np.array([1, 1]), "tokens": np.array([[1, 9, -1, -1], [4, 7, -1, -1]]),
                      "acc_margin": np.full((R, g), 1.0), "corr_margin": np.array([1.0, 1.0]),
                      "corr_rho": np.ones((R, 2))}}
    gpu = {"x": ref["draft"]["x"].copy(), "ell": ref["sched"]["ell"].copy(), "n_acc": ref["verify"]["n_acc"].copy(),
           "tokens": ref["verify"]["tokens"].copy()}
    c = bench.compare_round(gpu, ref)
    assert c["boundary_cases"] == 0 and c["mismatches"] == 0
    gpu["x"][1, 2] = 0
    ref["draft"]["margin"][1, 2] = 1e-6  # runner-up 0 within the boundary
    c = bench.compare_round(gpu, ref)
    assert c["boundary_cases"] == 1 and c["mismatches"] == 0
    gpu["tokens"][0, 1] = 8  # a correction token differing with a wide margin
    c = bench.compare_round(gpu, ref)
    assert c["mismatches"] == 1


def test_clock_summary_and_nvml_reason_bits():
    import bench
    assert bench.nvml_reason_names(0) == []
    assert bench.nvml_reason_names(0x4) == ["sw_power_cap"]
    assert set(bench.nvml_reason_names(0x8 | 0x20 | 0x40)) == {"hw_slowdown", "sw_thermal_slowdown",
                                                               "hw_thermal_slowdown"}
    assert bench.nvml_reason_names(0x80) == ["hw_slowdown"]  # HW power brake
    assert bench.nvml_reason_names(0x1 | 0x2) == []  # idle, application clocks: not throttling
    s = bench.summarize_clock_samples([(2070.0, 2070.0, []), (1950.0, 2070.0, ["sw_power_cap"]),
                                       (2070.0, 2070.0, [])])
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.summarize_clock_samples([])["reasons"] == ["unsampled"]


def test_clock_sampler_polls_nvml_from_a_thread(monkeypatch):
    """With an NVML device (a fake here: no driver on this machine) the sampler polls from a
    host thread for the whole region; without one it falls back and reports 'unsampled'."""
    import time
    import bench

    class FakeNvml:
        def __init__(self, index):
            self.n = 0

        def sample(self):
            self.n += 1
            return (2070.0 if self.n % 3 else 1980.0, 2070.0, ["sw_power_cap"] if self.n == 2 else [])

    monkeypatch.setattr(bench, "_NvmlClocks", FakeNvml)
    with bench.ClockSampler(0) as c:
        time.sleep(0.05)
    s = c.summary()
    assert s["source"] == "nvml" and s["samples"] >= 5
    assert s["sm_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]

    def no_nvml(index):
        raise OSError("libnvidia-ml.so.1: cannot open shared object file")

    monkeypatch.setattr(bench, "_NvmlClocks", no_nvml)
    monkeypatch.setenv("PATH", "/nonexistent")  # no nvidia-smi either
    with bench.ClockSampler(0) as c:
        pass
    assert c.summary()["reasons"] == ["unsampled"]
