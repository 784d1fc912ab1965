"""A round captured as a CUDA graph computes what the same round computes when its
calls are launched one by one (the library does no host work that capture would
freeze, and its programmatic-dependent launches keep their order inside a graph)."""
import pytest
import torch

from speculative_decoding_draft_03_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over", [("tiny", {}), ("qwen3-8b", dict(V=20000, d=256)),
                                       ("deepseek-v4", dict(V=4104, d=256))])
def test_graph_replay_matches_eager_round(name, over):
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make(name, device="cuda", **over)
    rd = b.Round(w)
    outs = []
    for rnd in (5, 6):
        d, s, v = rd.run(rnd=rnd)
        torch.cuda.synchronize()
        outs.append({k: t.clone() for k, t in {**d, **s, **v}.items()})
    graphs = [rd.capture(rnd=5), rd.capture(rnd=6)]
    for rep in range(2):  # replays are repeatable
        for i, g in enumerate(graphs):
            g.replay()
            torch.cuda.synchronize()
            got = {**rd.draft_out, **rd.sched_out, **rd.verify_out}
            for k, ref in outs[i].items():
                assert torch.equal(got[k], ref), (name, rep, i, k)
    assert rd.status() == 0


def test_graph_records_step_events():
    from speculative_decoding_draft_03_gb300 import binding as b
    w = wl.make("qwen3-8b", device="cuda", V=20000, d=256)
    rd = b.Round(w)
    timer = b.StepTimer(w["gamma"])
    g = rd.capture(rnd=1, timer=timer)
    g.replay()
    torch.cuda.synchronize()
    timer.collect()
    assert len(timer.samples) == w["gamma"]
    assert all(0.0 < t < 100.0 for t in timer.samples)
