"""One batch of R requests split over the ranks of a process group, with one global
confidence scheduler.

Requests are independent in the draft and verification stages, so each rank drafts and
verifies its own contiguous slice of the batch (its request ids are the batch's, so its
draws are exactly those of the unsplit batch).  The scheduler is global: it sorts every
(request, depth) candidate of the batch by its survival product and walks the verify
budget against SPS(B) (numb3r33 blog "Greedy prefix allocation"; DSpark 精读 §4).  So
the ranks exchange their confidences once per round, an all-gather of the [R, gamma]
fp32 confidences (30 KB at R = 512, gamma = 15), every rank runs the same scheduler on
the whole batch, and each keeps its own slice of the verify lengths.  B and tau are the
whole batch's on every rank.

On GPUs the all-gather is a torch.distributed (NCCL) collective enqueued on the current
stream between the draft and the scheduler; nothing else is exchanged.  The host-side
pieces (partition, gather, slice) run unchanged on CPU process groups (gloo).
"""
from __future__ import annotations

import torch


def partition(R: int, world: int, rank: int):
    """Contiguous slice [lo, hi) of the R requests owned by `rank`: the first R % world
    ranks take one request more."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a group of {world}")
    base, extra = divmod(R, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def gather_confidences(conf_local: torch.Tensor, R: int, world: int, group=None) -> torch.Tensor:
    """All-gather of the ranks' confidence slices [hi - lo, gamma] into the batch's
    [R, gamma], in request order.  Slices are padded to a common row count for the
    collective and the padding is dropped."""
    import torch.distributed as dist
    gamma = conf_local.shape[1]
    if world == 1:
        return conf_local
    rows = -(-R // world)
    buf = torch.zeros((rows, gamma), dtype=conf_local.dtype, device=conf_local.device)
    buf[:conf_local.shape[0]].copy_(conf_local)
    full = torch.empty((world * rows, gamma), dtype=conf_local.dtype, device=conf_local.device)
    dist.all_gather_into_tensor(full, buf, group=group)
    parts = []
    for r in range(world):
        lo, hi = partition(R, world, r)
        parts.append(full[r * rows:r * rows + (hi - lo)])
    return torch.cat(parts, 0).contiguous()


class ShardedRound:
    """This rank's share of one DSpark round over a batch split across `world` ranks.

    `w` is the whole batch's workload (its per-request tensors are sliced to this rank's
    requests; the weights are shared).  run() drafts this rank's requests, gathers every
    rank's confidences, runs the scheduler on the whole batch, and verifies this rank's
    requests with their slice of the verify lengths.  `gather` replaces the collective
    (a callable conf_local -> conf_full), e.g. to run several ranks' shares in one
    process."""

    PER_REQUEST = ("U", "target", "h", "x0", "req_id")

    def __init__(self, w: dict, world: int, rank: int, group=None, gather=None):
        from . import binding as b
        self.b = b
        self.R_total = w["R"]
        self.world, self.rank, self.group = world, rank, group
        self.lo, self.hi = partition(self.R_total, world, rank)
        local = dict(w)
        for k in self.PER_REQUEST:
            local[k] = w[k][self.lo:self.hi].contiguous()
        local["R"] = self.hi - self.lo
        self.w = local
        self.full = w
        self._gather = gather
        R, gamma, V, rank_, d = local["R"], w["gamma"], w["V"], w["rank"], w["d"]
        dev = w["U"].device
        self.draft_out = dict(x=torch.empty((R, gamma), dtype=torch.int32, device=dev),
                              logq=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                              lse=torch.empty((R, gamma), dtype=torch.float32, device=dev),
                              conf=torch.empty((R, gamma), dtype=torch.float32, device=dev))
        self.sched_out = dict(ell=torch.empty(self.R_total, dtype=torch.int32, device=dev),
                              B=torch.empty(1, dtype=torch.int32, device=dev),
                              tau=torch.empty(1, dtype=torch.float64, device=dev))
        self.verify_out = dict(n_acc=torch.empty(R, dtype=torch.int32, device=dev),
                               tokens=torch.empty((R, gamma + 1), dtype=torch.int32, device=dev),
                               n_out=torch.empty(R, dtype=torch.int32, device=dev))
        self.ws_draft = b.workspace(b.draft_workspace_size(R, gamma, V, rank_, d, w["W1"].dtype), dev)
        self.ws_sched = b.workspace(b.schedule_workspace_size(self.R_total, gamma), dev)
        self.ws_verify = b.workspace(b.verify_workspace_size(R, gamma, V, rank_, w["W1"].dtype), dev)

    def gather(self, conf_local):
        if self._gather is not None:
            return self._gather(conf_local)
        return gather_confidences(conf_local, self.R_total, self.world, self.group)

    def draft(self, rnd=0, x0=None, stream=None):
        b, w = self.b, self.w
        x0 = w["x0"] if x0 is None else x0
        return b.markov_draft(w["U"], w["W1"], w["W2"], w["h"], w["conf_w"], w["conf_b"], w["conf_logit_scale"],
                              w["conf_temp"], w["temperature"], x0, w["req_id"], w["seed"], rnd,
                              out=self.draft_out, ws=self.ws_draft, stream=stream)

    def schedule_and_verify(self, conf_full, rnd=0, x0=None, stream=None):
        """The global scheduler on the whole batch's confidences, then verification of this
        rank's requests with their slice of the verify lengths."""
        b, w, full = self.b, self.w, self.full
        x0 = w["x0"] if x0 is None else x0
        s = b.schedule(conf_full, full["sps"], full["mode"], full.get("conf_hist"), full.get("fixed_len", 0),
                       out=self.sched_out, ws=self.ws_sched, stream=stream)
        ell = s["ell"][self.lo:self.hi]
        d = self.draft_out
        v = b.verify(w["target"], w["U"], w["W1"], w["W2"], x0, d["x"], d["logq"], d["lse"], ell, w["temperature"],
                     w["req_id"], w["seed"], rnd, out=self.verify_out, ws=self.ws_verify, stream=stream)
        return s, v

    def run(self, rnd=0, x0=None, stream=None):
        d = self.draft(rnd, x0, stream)
        conf_full = self.gather(d["conf"])
        s, v = self.schedule_and_verify(conf_full, rnd, x0, stream)
        return d, s, v
