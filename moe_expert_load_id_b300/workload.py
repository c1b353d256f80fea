"""Seeded synthetic inputs for the balancing hot path.

This module holds no step of the method: it only draws the gate's top-k expert
ids and the bf16 hidden rows.  Both the CUDA path and the CPU oracle are fed
from here.

Workloads stand in for the pages' real routing traces (Megatron-LM training
and SGLang prefill on Qwen3-235B, GLM-4.5 and DeepSeek-V3; UltraEP article,
evaluation paragraph), which are not available: the shapes (ranks, experts,
spare slots, top-k, tokens, layers, hidden size) follow those models, and the
expert popularity is synthetic.

Recipe
------
* Popularity p[e] of one (layer, microbatch) is drawn on the host with numpy
  PCG64 from the seed ``base + 1000*layer + microbatch`` (base per workload):
  - ``zipf``:  p[e] proportional to 1 / (pi[e] + 1)**s over a seeded random
    permutation pi of the experts (per layer, or per (layer, microbatch) when
    ``redraw`` is set);
  - ``dirichlet_drift``: p = 0.5*d_l + 0.5*((1 - m/(M-1))*A_l + (m/(M-1))*B_l)
    with d_l, A_l, B_l ~ Dirichlet(alpha) fixed per layer and m the microbatch.
* Each token draws k DISTINCT experts by Gumbel-top-k: the k largest of
  log p[e] + G[e], G = -log(-log U), U ~ Uniform[0, 1) in float64, drawn with a
  torch generator seeded from the same seed (on the host or on the device;
  the two generators give different, equally valid, draws).  The k ids of a
  token are listed by descending score, as a gate's top-k is.
* Hidden rows are N(0, 1) float32 rounded to bf16 (round to nearest even),
  from a torch generator seeded with ``seed + 7``.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    R: int          # ranks of the simulated EP domain
    E: int          # logical experts
    S: int          # spare slots per rank
    k: int          # top-k
    T: int          # tokens per microbatch over the whole domain
    layers: int
    microbatches: int
    Hd: int         # hidden size (bf16 elements per row)
    popularity: str = "zipf"
    s: float = 1.0
    alpha: float = 0.3
    redraw: bool = False
    base_seed: int = 20261202

    @property
    def H(self) -> int:
        return self.E // self.R

    @property
    def P(self) -> int:
        return self.R * (self.H + self.S)

    @property
    def N(self) -> int:
        return self.T * self.k

    def seed(self, layer: int, microbatch: int) -> int:
        return self.base_seed + 1000 * layer + microbatch

    def domain(self):
        return dict(R=self.R, E=self.E, S=self.S, k=self.k)

    def popularity_desc(self) -> str:
        if self.popularity == "dirichlet_drift":
            return (f"popularity 0.5 Dirichlet({self.alpha}) per layer + 0.5 drift between two "
                    f"Dirichlet({self.alpha}) endpoints over {self.microbatches} microbatches")
        when = "re-drawn every microbatch" if self.redraw else "fixed per layer"
        return f"Zipf(s={self.s}) popularity {when}"


WORKLOADS = {
    "tiny": Workload("tiny", R=8, E=32, S=1, k=4, T=4096, layers=4, microbatches=1,
                     Hd=256, popularity="zipf", s=1.2, base_seed=11_000_000),
    "qwen3-235b": Workload("qwen3-235b", R=64, E=128, S=1, k=8, T=64 * 2048, layers=94,
                           microbatches=4, Hd=4096, popularity="zipf", s=1.0, redraw=True,
                           base_seed=12_000_000),
    "deepseek-v3": Workload("deepseek-v3", R=64, E=256, S=2, k=8, T=64 * 2048, layers=58,
                            microbatches=16, Hd=7168, popularity="dirichlet_drift",
                            alpha=0.3, base_seed=13_000_000),
    "glm-4.5": Workload("glm-4.5", R=40, E=160, S=1, k=8, T=40 * 4096, layers=89,
                        microbatches=4, Hd=5120, popularity="zipf", s=1.4,
                        base_seed=14_000_000),
}


def stress(R: int, S: int, tokens_per_rank: int, s: float) -> Workload:
    """One point of the stress sweep: E = 4R, k = 8, hidden 4096, 32 layers."""
    return Workload(f"stress-R{R}-S{S}-T{tokens_per_rank}-s{s}", R=R, E=4 * R, S=S, k=8,
                    T=tokens_per_rank * R, layers=32, microbatches=1, Hd=4096,
                    popularity="zipf", s=s, base_seed=15_000_000 + 1000 * R + 10 * S)


STRESS_GRID = dict(R=(8, 16, 32, 64), S=(1, 2, 4), tokens_per_rank=(512, 1024, 2048, 4096, 8192),
                   s=(0.6, 1.0, 1.6))


def popularity(w: Workload, layer: int, microbatch: int) -> np.ndarray:
    """Expert popularity p[E] (float64, sums to 1) of one (layer, microbatch)."""
    if w.popularity == "zipf":
        key = w.seed(layer, microbatch if w.redraw else 0)
        rng = np.random.Generator(np.random.PCG64(key))
        perm = rng.permutation(w.E)
        p = 1.0 / (perm + 1.0) ** w.s
    elif w.popularity == "dirichlet_drift":
        rng = np.random.Generator(np.random.PCG64(w.seed(layer, 0)))
        a = np.full(w.E, w.alpha)
        d, A, B = rng.dirichlet(a), rng.dirichlet(a), rng.dirichlet(a)
        f = microbatch / max(1, w.microbatches - 1)
        p = 0.5 * d + 0.5 * ((1.0 - f) * A + f * B)
    elif w.popularity == "uniform":
        p = np.ones(w.E)
    else:
        raise ValueError(w.popularity)
    return p / p.sum()


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gumbel_topk(p: np.ndarray, T: int, k: int, seed: int, device="cpu",
                chunk: int = 1 << 15) -> torch.Tensor:
    """[T, k] int32: k distinct expert ids per token, by Gumbel-top-k over log p."""
    E = len(p)
    if k > E:
        raise ValueError("k > E")
    logp = torch.from_numpy(np.log(np.maximum(p, 1e-300))).to(device=device, dtype=torch.float64)
    g = _gen(seed, device)
    out = torch.empty((T, k), dtype=torch.int32, device=device)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        u = torch.rand((t1 - t0, E), generator=g, dtype=torch.float64, device=device)
        score = logp[None, :] - torch.log(-torch.log(u))
        out[t0:t1] = torch.topk(score, k, dim=1, largest=True, sorted=True).indices.to(torch.int32)
    return out


def topk_ids(w: Workload, layer: int, microbatch: int, device="cpu") -> torch.Tensor:
    """The gate's top-k ids [T, k] int32 of one (layer, microbatch)."""
    return gumbel_topk(popularity(w, layer, microbatch), w.T, w.k, w.seed(layer, microbatch),
                       device=device)


def hidden(T: int, Hd: int, seed: int, device="cpu", chunk_rows: int = 1 << 14) -> torch.Tensor:
    """[T, Hd] bf16 rows drawn from N(0, 1)."""
    g = _gen(seed + 7, device)
    out = torch.empty((T, Hd), dtype=torch.bfloat16, device=device)
    for t0 in range(0, T, chunk_rows):
        t1 = min(T, t0 + chunk_rows)
        out[t0:t1] = torch.randn((t1 - t0, Hd), generator=g, dtype=torch.float32,
                                 device=device).to(torch.bfloat16)
    return out


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a bf16 tensor, as a host uint16 array."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
