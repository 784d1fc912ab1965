"""bench.py's command line and the pieces of its JSON line that need no GPU: the options
parse, every workload has a description, and the stored draft-step traffic is read only
when the profile was taken on the current kernel source."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_help_lists_every_mode():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr
    for opt in ("--gpus", "--steps", "--warmup", "--impl", "--workload", "--head", "--diagnostic"):
        assert opt in r.stdout, opt
    for mode in ("overlap", "verify_overlap", "sts"):
        assert mode in r.stdout, mode


def test_workload_descriptions_and_stored_traffic():
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_draft_03_gb300 import workloads as wl
    for name in wl.SHAPES:
        assert bench.WORKLOAD_DESC[name]
    t = bench.stored_traffic("qwen3-8b")
    # either the committed profile matches the kernel source (then its DRAM bytes are
    # about the algorithmic 97.26 MB per launch), or the traffic is reported as unknown
    assert t is None or 90e6 < t < 110e6, t
