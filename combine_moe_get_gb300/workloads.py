"""Seeded synthetic workloads for MoE layout / dispatch / combine.

This module only draws random inputs: token hidden rows, top-k expert choices,
router weights and expert-side partial rows. It holds none of the routing,
counting, copying or reduction arithmetic of the method itself, so that the
CUDA path and the CPU oracle can both be fed from it without sharing any of
that arithmetic.

Every draw uses a CPU ``torch.Generator`` seeded per workload, so the inputs
do not depend on the GPU. Draw order within a workload is fixed:
hidden rows ``x``, then top-k keys, then router logits, then partial rows.

Workload shapes follow the DeepEP V2 deep-dive page ("DeepEP V2 深度深潜",
section 1.3 and 2.2): ``num_experts`` experts spread evenly over ``num_ranks``
ranks (``E % R == 0``), ``num_topk <= 32`` choices per token, ``-1`` marking a
masked choice.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

__all__ = ["Workload", "CONFIGS", "Inputs", "make_inputs", "make_topk_uniform",
           "make_topk_zipf", "make_weights", "make_x", "make_partial",
           "mask_random_lanes", "recv_capacity"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_tokens: int
    hidden: int            # 0 for layout-only workloads
    num_experts: int
    num_ranks: int
    num_topk: int
    routing: str = "uniform"   # "uniform" (without replacement) or "zipf"
    zipf_s: float = 1.0
    fp8: bool = False          # dispatch quantises x to e4m3 with per-128 scales
    seed: int = 0

    @property
    def experts_per_rank(self) -> int:
        return self.num_experts // self.num_ranks

    @property
    def layout_only(self) -> bool:
        return self.hidden == 0


# The five workloads of the benchmark spec plus the layout-only 2048-expert run.
CONFIGS = {
    "tiny": Workload("tiny", 128, 256, 16, 4, 2),
    "dsv3": Workload("dsv3", 4096, 7168, 256, 8, 8),
    "dsv3_fp8": Workload("dsv3_fp8", 4096, 7168, 256, 8, 8, fp8=True),
    "skewed": Workload("skewed", 8192, 7168, 256, 64, 8, routing="zipf", zipf_s=1.0),
    "decode": Workload("decode", 128, 7168, 256, 256, 8),
    "layout_2048": Workload("layout_2048", 128, 0, 2048, 256, 8),
    "layout_2048_1m": Workload("layout_2048_1m", 1 << 20, 0, 2048, 256, 8),
}


def recv_capacity(num_tokens: int, num_topk: int, num_ranks: int) -> int:
    """Worst-case number of received rows: every token reaches min(k, R) ranks."""
    return num_tokens * min(num_topk, num_ranks)


def make_x(gen: torch.Generator, num_tokens: int, hidden: int) -> torch.Tensor:
    """Hidden rows ~ N(0, 1) drawn in fp32, rounded to bf16 (torch's RNE cast)."""
    return torch.randn(num_tokens, hidden, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_topk_uniform(gen: torch.Generator, num_tokens: int, num_experts: int,
                      num_topk: int) -> torch.Tensor:
    """k distinct experts per token, uniform over k-subsets.

    Sequential sampling without replacement: column j is drawn uniformly and
    re-drawn wherever it repeats an earlier column of the same row, which makes
    it uniform over the experts not yet chosen in that row.
    """
    if num_topk > num_experts:
        raise ValueError("num_topk > num_experts")
    out = torch.empty(num_tokens, num_topk, dtype=torch.int64)
    for j in range(num_topk):
        col = torch.randint(0, num_experts, (num_tokens,), generator=gen, dtype=torch.int64)
        while j > 0:
            clash = (out[:, :j] == col[:, None]).any(dim=1)
            n = int(clash.sum())
            if n == 0:
                break
            col[clash] = torch.randint(0, num_experts, (n,), generator=gen, dtype=torch.int64)
        out[:, j] = col
    return out


def make_topk_zipf(gen: torch.Generator, num_tokens: int, num_experts: int,
                   num_topk: int, s: float) -> torch.Tensor:
    """k distinct experts per token with Zipf(s) popularity.

    Expert e has weight 1 / pi(e)^s for a random permutation pi of 1..E; the k
    experts are drawn without replacement proportionally to these weights via
    Gumbel-top-k (perturb log-weights with Gumbel noise, keep the k largest).
    """
    perm = torch.randperm(num_experts, generator=gen) + 1
    logw = -s * torch.log(perm.to(torch.float64))
    u = torch.rand(num_tokens, num_experts, generator=gen, dtype=torch.float64)
    u = u.clamp_min(1e-300)
    gumbel = -torch.log(-torch.log(u))
    keys = logw[None, :] + gumbel
    return torch.topk(keys, num_topk, dim=1).indices.to(torch.int64)


def make_weights(gen: torch.Generator, num_tokens: int, num_topk: int) -> torch.Tensor:
    """Router weights: softmax of N(0, 1) logits, fp32 [T, k]."""
    logits = torch.randn(num_tokens, num_topk, generator=gen, dtype=torch.float32)
    return torch.softmax(logits, dim=1)


def make_partial(gen: torch.Generator, rows: int, hidden: int) -> torch.Tensor:
    """Expert-side partial rows ~ N(0, 1) in bf16, [rows, H]."""
    return torch.randn(rows, hidden, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def mask_random_lanes(gen: torch.Generator, topk_idx: torch.Tensor, frac: float) -> torch.Tensor:
    """Copy of ``topk_idx`` with about ``frac`` of its entries set to -1 (masked)."""
    m = torch.rand(topk_idx.shape, generator=gen) < frac
    out = topk_idx.clone()
    out[m] = -1
    return out


@dataclasses.dataclass
class Inputs:
    workload: Workload
    x: Optional[torch.Tensor]          # [T, H] bf16, None for layout-only
    topk_idx: torch.Tensor             # [T, k] int64
    topk_weights: torch.Tensor         # [T, k] fp32
    partial: Optional[torch.Tensor]    # [capacity, H] bf16, None unless requested


def make_inputs(w: Workload, with_partial: bool = True, num_tokens: Optional[int] = None) -> Inputs:
    """All inputs of workload ``w`` (CPU tensors), drawn in the fixed order.

    ``num_tokens`` overrides the token count (for reduced-size cases); the
    partial rows cover the worst-case receive capacity so that their shape does
    not depend on the routing.
    """
    T = w.num_tokens if num_tokens is None else num_tokens
    gen = torch.Generator().manual_seed(w.seed)
    x = None if w.layout_only else make_x(gen, T, w.hidden)
    if w.routing == "uniform":
        topk = make_topk_uniform(gen, T, w.num_experts, w.num_topk)
    elif w.routing == "zipf":
        topk = make_topk_zipf(gen, T, w.num_experts, w.num_topk, w.zipf_s)
    else:
        raise ValueError(w.routing)
    weights = make_weights(gen, T, w.num_topk)
    partial = None
    if with_partial and not w.layout_only:
        partial = make_partial(gen, recv_capacity(T, w.num_topk, w.num_ranks), w.hidden)
    return Inputs(w, x, topk, weights, partial)

