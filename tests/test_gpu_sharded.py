"""The split-batch round (speculative_decoding_draft_03_gb300/sharded.py) on the GPU:
the shares of two and three ranks, run one after the other in one process (the
collective replaced by concatenation of the shares' confidences), give exactly the
unsplit round's drafts, verify lengths, B, tau and tokens."""
import pytest
import torch

from speculative_decoding_draft_03_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over,world", [("qwen3-8b", dict(V=20000, d=256), 2),
                                             ("deepseek-v4", dict(V=4104, d=256), 3),
                                             ("tiny", {}, 2)])
def test_split_batch_equals_unsplit_round(name, over, world):
    from speculative_decoding_draft_03_gb300 import binding as b
    from speculative_decoding_draft_03_gb300.sharded import ShardedRound
    w = wl.make(name, device="cuda", **over)
    rnd = 4
    d, s, v = b.Round(w).run(rnd=rnd)
    shares = [ShardedRound(w, world, r, gather=lambda c: None) for r in range(world)]
    drafts = [sh.draft(rnd) for sh in shares]
    conf_full = torch.cat([dd["conf"] for dd in drafts], 0)
    outs = [sh.schedule_and_verify(conf_full, rnd) for sh in shares]
    torch.cuda.synchronize()
    for k in ("x", "logq", "lse", "conf"):
        assert torch.equal(torch.cat([dd[k] for dd in drafts], 0), d[k]), k
    for ss, _ in outs:
        assert torch.equal(ss["ell"], s["ell"]) and torch.equal(ss["B"], s["B"]) and torch.equal(ss["tau"], s["tau"])
    for k in ("n_acc", "tokens", "n_out"):
        assert torch.equal(torch.cat([vv[k] for _, vv in outs], 0), v[k]), k
