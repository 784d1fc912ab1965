"""Seeded synthetic workloads for the DSpark per-round hot path.

This module holds only input recipes: shapes, distributions, seeds, and the profiled
step-rate tables SPS(B).  It contains none of the method's arithmetic, so both the
CUDA library's tests/benchmark and the CPU oracle draw their inputs from here.

Recipes (the five workloads of the draft/schedule/verify path):

* ``tiny``        R=4, gamma=4, V=1024, rank=32, d=64, everything fp32.
                  U ~ N(0,2^2); W1, W2 ~ N(0,0.1^2); target = U + N(0,0.5^2) over gamma+1
                  rows (row gamma reuses U's last row); h ~ N(0,1); confidence weights
                  ~ N(0,0.05^2); SPS(B) = 1000/(1+B/64); early-stop scheduler.
* ``qwen3-8b``    R=32, gamma=7, V=151936, rank=256, d=4096.  U fp32 ~ N(0,3^2) plus a
                  Zipf(1.1) log-prior -1.1*ln(v+1) (rank = token id); W1, W2 bf16
                  ~ N(0,0.02^2); target = U + N(0, sigma_k^2), sigma_k = 0.3+0.1k for
                  k = 1..gamma+1; h bf16; SPS flat (1000) up to B=64, then 1000*64/B.
* ``batch128``    R=128, gamma=16, same dims/distributions as qwen3-8b; SPS a step table
                  S0*0.88^n, n = number of {128,256,512,1024} strictly below B;
                  full-search scheduler (jagged table).
* ``deepseek-v4`` R=256, gamma=5, V=129280, rank=256, d=4096.  U and target bf16,
                  target = U + N(0,0.4^2); confidence logits scaled by 1.5
                  (overconfident); SPS steps at 256/512/1024/1536 with 12% drops;
                  capacity-K scheduler whose K comes from a second, independently
                  seeded confidence set standing for the round two back.
* ``stress``      R=512, gamma=15, V=151936, rank=256, d=4096, logits fp32, weights bf16;
                  per-request target noise sigma in {0.1, 0.5, 1.5} for 200/200/112
                  requests (a seeded permutation assigns them); SPS linear then a cliff:
                  S0*(1-0.2*B/2048) up to B=2048, half that value just past it, then
                  falling as 1/B; early-stop scheduler; 100 chained rounds.

Any workload can be drafted by the recurrent head instead (``add_rnn_head``).

All workloads: anchor x0 ~ U[0,V), request ids 0..R-1, sampling seed 0, T = 1, STS
temperatures 1, confidence bias 0.  Each tensor has its own torch.Generator seed, so a
workload is reproducible on a given device type.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

EARLY_STOP, FULL_SEARCH, CAPACITY_K, FIXED = 0, 1, 2, 3
S0 = 1000.0


@dataclass(frozen=True)
class Shape:
    name: str
    R: int
    gamma: int
    V: int
    rank: int
    d: int
    u_dtype: torch.dtype
    t_dtype: torch.dtype
    w_dtype: torch.dtype
    h_dtype: torch.dtype
    mode: int
    kappa: float = 1.0
    rounds: int = 1
    extra: dict = field(default_factory=dict)


SHAPES = {
    "tiny": Shape("tiny", 4, 4, 1024, 32, 64, torch.float32, torch.float32, torch.float32,
                  torch.float32, EARLY_STOP),
    "qwen3-8b": Shape("qwen3-8b", 32, 7, 151936, 256, 4096, torch.float32, torch.float32,
                      torch.bfloat16, torch.bfloat16, EARLY_STOP),
    "batch128": Shape("batch128", 128, 16, 151936, 256, 4096, torch.float32, torch.float32,
                      torch.bfloat16, torch.bfloat16, FULL_SEARCH),
    "deepseek-v4": Shape("deepseek-v4", 256, 5, 129280, 256, 4096, torch.bfloat16,
                         torch.bfloat16, torch.bfloat16, torch.bfloat16, CAPACITY_K, kappa=1.5),
    "stress": Shape("stress", 512, 15, 151936, 256, 4096, torch.float32, torch.float32,
                    torch.bfloat16, torch.bfloat16, EARLY_STOP, rounds=100),
}


def sps_table(name: str, R: int, gamma: int) -> np.ndarray:
    """Profiled target steps/s as a function of the verify batch B = sum_r (1 + l_r)."""
    n = R * (gamma + 1) + 1
    B = np.arange(n, dtype=np.float64)
    if name == "tiny":
        return S0 / (1.0 + B / 64.0)
    if name == "qwen3-8b":
        return np.where(B <= 64, S0, S0 * 64.0 / np.maximum(B, 1.0))
    if name == "batch128":
        steps = sum((B > s).astype(np.float64) for s in (128, 256, 512, 1024))
        return S0 * 0.88 ** steps
    if name == "deepseek-v4":
        steps = sum((B > s).astype(np.float64) for s in (256, 512, 1024, 1536))
        return S0 * 0.88 ** steps
    if name == "stress":
        at_cliff = S0 * (1.0 - 0.2)
        return np.where(B <= 2048, S0 * (1.0 - 0.2 * B / 2048.0),
                        0.5 * at_cliff * 2048.0 / np.maximum(B, 1.0))
    raise KeyError(name)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, sigma, seed, device, out_dtype=torch.float32):
    t = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    t.mul_(sigma)
    return t.to(out_dtype) if out_dtype != torch.float32 else t


def make(name: str, device="cpu", seed: int = 0, **override) -> dict:
    """Generate one workload.  Tensors live on ``device``; scalars are Python numbers.

    ``override`` may replace R, gamma, V, rank, d (shrunken variants for fast tests keep
    the named workload's distributions).
    """
    sh = SHAPES[name]
    R = override.get("R", sh.R)
    gamma = override.get("gamma", sh.gamma)
    V = override.get("V", sh.V)
    rank = override.get("rank", sh.rank)
    d = override.get("d", sh.d)
    base = 1000 * (seed + 1)
    dev = torch.device(device)

    if name == "tiny":
        u_sigma, w_sigma, zipf = 2.0, 0.1, 0.0
    else:
        u_sigma, w_sigma, zipf = 3.0, 0.02, 1.1

    U = _normal((R, gamma, V), u_sigma, base + 1, dev)
    if zipf:
        prior = -zipf * torch.log(torch.arange(V, device=dev, dtype=torch.float32) + 1.0)
        U.add_(prior)
    # target rows k = 1..gamma+1 use U row min(k, gamma) (1-indexed)
    src = torch.cat([U, U[:, gamma - 1:gamma, :]], dim=1)
    noise = torch.randn((R, gamma + 1, V), generator=_gen(dev, base + 2), device=dev,
                        dtype=torch.float32)
    if name == "tiny":
        sig = torch.full((R, gamma + 1, 1), 0.5, device=dev)
    elif name == "deepseek-v4":
        sig = torch.full((R, gamma + 1, 1), 0.4, device=dev)
    elif name == "stress":
        perm = torch.randperm(R, generator=_gen("cpu", base + 3))
        n1 = round(R * 200 / 512)
        n2 = round(R * 400 / 512)
        cls = torch.empty(R)
        cls[perm[:n1]] = 0.1
        cls[perm[n1:n2]] = 0.5
        cls[perm[n2:]] = 1.5
        sig = cls.to(dev).view(R, 1, 1).expand(R, gamma + 1, 1)
    else:
        k = torch.arange(1, gamma + 2, device=dev, dtype=torch.float32)
        sig = (0.3 + 0.1 * k).view(1, gamma + 1, 1).expand(R, gamma + 1, 1)
    target = src + noise * sig
    del src, noise
    U = U.to(sh.u_dtype)
    target = target.to(sh.t_dtype)

    W1 = _normal((V, rank), w_sigma, base + 4, dev, sh.w_dtype)
    W2 = _normal((rank, V), w_sigma, base + 5, dev, sh.w_dtype)
    h = _normal((R, gamma, d), 1.0, base + 6, dev, sh.h_dtype)
    conf_w = _normal((d + rank,), 0.05, base + 7, dev)
    x0 = torch.randint(0, V, (R,), generator=_gen(dev, base + 8), device=dev, dtype=torch.int64).to(torch.int32)
    req_id = torch.arange(R, device=dev, dtype=torch.int64)
    conf_temp = torch.ones(gamma, device=dev, dtype=torch.float32)
    out = dict(name=name, R=R, gamma=gamma, V=V, rank=rank, d=d, U=U, target=target, W1=W1,
               W2=W2, h=h, conf_w=conf_w, conf_b=0.0, conf_logit_scale=sh.kappa,
               conf_temp=conf_temp, temperature=1.0, x0=x0, req_id=req_id, seed=0,
               mode=sh.mode, fixed_len=0, rounds=sh.rounds,
               sps=torch.from_numpy(sps_table(name, R, gamma)).to(dev))
    if sh.mode == CAPACITY_K:
        # stale confidences of the round two back: same logit law as the live head
        # (w.h with w ~ N(0,0.05^2), h ~ N(0,1) gives N(0, d*0.05^2)), scaled by kappa
        z = _normal((R, gamma), math.sqrt(d) * 0.05, base + 9, dev)
        out["conf_hist"] = torch.sigmoid(sh.kappa * z).to(torch.float32)
    else:
        out["conf_hist"] = None
    return out


def add_rnn_head(w: dict, seed: int = 0) -> dict:
    """The same workload drafted by the recurrent head: state width ns = rank, embedding
    width ne = rank, weights in the workload's weight type.  E ~ N(0,1);
    Wse ~ N(0, 1/(ns+ne)); Wh ~ N(0, 0.25/d); gate bias -1 (the gate starts mostly
    shut), candidate bias 0; Wo ~ N(0, 0.02^2) like the Markov factors.  The confidence
    weights' last ns entries apply to the state.  W1/W2 are dropped."""
    dev = w["U"].device
    wdt = w["W1"].dtype
    ns = ne = w["rank"]
    V, d = w["V"], w["d"]
    base = 1000 * (seed + 1) + 20
    out = dict(w)
    out.pop("W1")
    out.pop("W2")
    out["head"] = "rnn"
    out["ns"], out["ne"] = ns, ne
    out["E"] = _normal((V, ne), 1.0, base + 1, dev, wdt)
    out["Wse"] = _normal((ns + ne, 2 * ns), 1.0 / math.sqrt(ns + ne), base + 2, dev, wdt)
    out["Wh"] = _normal((d, 2 * ns), 0.5 / math.sqrt(max(d, 1)), base + 3, dev, wdt)
    out["bgc"] = torch.cat([torch.full((ns,), -1.0, device=dev), torch.zeros(ns, device=dev)])
    out["Wo"] = _normal((ns, V), 0.02, base + 4, dev, wdt)
    return out


def sts_heldout(N: int, gamma: int, T_true, seed: int = 0, mu: float = 1.5, sigma: float = 2.0,
                device="cpu") -> dict:
    """Synthetic held-out rounds for fitting the per-position temperatures: confidence
    logits z[n,k] ~ N(mu, sigma^2) and accepted lengths drawn from a known calibration
    law, position k surviving with probability sigmoid(z[n,k] / T_true[k]) given that
    position k-1 survived (L = survivors before the first failure).  The fitted
    temperatures should come out near T_true."""
    dev = torch.device(device)
    z = _normal((N, gamma), sigma, 7000 + seed, dev).add_(mu)
    u = torch.rand((N, gamma), generator=_gen(dev, 7100 + seed), device=dev)
    T = torch.as_tensor(np.asarray(T_true, np.float32), device=dev).view(1, gamma)
    alive = (u < torch.sigmoid(z / T)).to(torch.int32)
    L = torch.cumprod(alive, dim=1).sum(dim=1).to(torch.int32)
    return dict(z=z, acc_len=L, T_true=np.asarray(T_true, np.float64))


def sts_grid(G: int = 256, lo: float = 0.05, hi: float = 20.0) -> np.ndarray:
    """Candidate temperatures, log-spaced."""
    return np.exp(np.linspace(math.log(lo), math.log(hi), G)).astype(np.float32)


def to_numpy(w: dict) -> dict:
    """Host copies for the oracle: bf16 tensors become their raw uint16 bit patterns."""
    out = {}
    for k, v in w.items():
        if isinstance(v, torch.Tensor):
            t = v.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                out[k] = t.view(torch.int16).numpy().view(np.uint16)
            else:
                out[k] = t.numpy()
        else:
            out[k] = v
    return out


def subset(wn: dict, rows) -> dict:
    """The per-request slice of a host workload (requests are independent in the draft
    and verify stages; the weights are shared)."""
    rows = np.asarray(rows)
    out = dict(wn)
    for k in ("U", "target", "h", "x0", "req_id"):
        out[k] = np.ascontiguousarray(wn[k][rows])
    out["R"] = len(rows)
    return out
