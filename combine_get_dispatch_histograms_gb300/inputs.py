"""Seeded synthetic inputs for MoE expert-parallel dispatch / combine.

This module only draws random numbers: it holds none of the dispatch or
combine arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.

Every workload is R virtual ranks, each holding T tokens of hidden size H
(bf16), a router choice ``topk_idx [R][T][K]`` (int64, -1 = masked) over E
experts and ``topk_weights [R][T][K]`` (fp32).  The five workloads follow the
shapes named for this method (a small worked case, a prefill batch, a decode
batch, a Zipf-skewed batch with masking, and a 4-node hierarchical batch).

Router recipes (the router itself is not part of the dispatch path):

* ``normal``: logits ~ N(0, 1); top-K of the logits (distinct experts);
  weights = softmax over the K chosen logits (renormalised, fp32).
* ``bias``:   as ``normal`` plus a per-expert bias ~ N(0, bias_std) shared by
  all tokens, which makes some experts popular.
* ``zipf``:   expert popularity p_i proportional to 1 / rank_i^s over a random
  permutation of the experts; K distinct experts drawn without replacement
  with probability proportional to p (Gumbel-top-K on log p + Gumbel noise);
  weights = softmax over the chosen perturbed logits; each entry is then masked
  to -1 independently with probability ``mask_p``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int            # virtual ranks
    E: int            # experts (E % R == 0, expert e lives on rank e // (E // R))
    K: int            # top-k
    T: int            # tokens per source rank
    H: int            # hidden size (bf16 channels)
    router: str = "normal"
    bias_std: float = 0.0
    zipf_s: float = 0.0
    mask_p: float = 0.0
    num_channels: int = 8
    num_nodes: int = 1
    ll_cap: int = 0   # low-latency tokens per (expert, source) region, 0 = not run in LL mode

    @property
    def L(self) -> int:
        return self.E // self.R

    @property
    def tokens(self) -> int:
        return self.R * self.T

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # R=4, E=8 (2 experts per rank), top-2: the worked case's shape.
    "tiny": Workload("tiny", R=4, E=8, K=2, T=16, H=128, router="normal", num_channels=2),
    # High-throughput prefill batch.
    "prefill": Workload("prefill", R=8, E=256, K=8, T=4096, H=7168, router="bias", bias_std=0.5),
    # Low-latency decode batch: T equals the per-rank dispatch cap.
    "decode": Workload("decode", R=16, E=256, K=8, T=128, H=7168, router="normal", ll_cap=128),
    # Zipf-skewed popularity with 5 % masked entries; LL runs in 256-token microbatches.
    "skewed": Workload("skewed", R=32, E=256, K=8, T=2048, H=4096, router="zipf", zipf_s=1.2,
                       mask_p=0.05, ll_cap=256),
    # 4 virtual nodes x 8 virtual ranks, hierarchical (node then rank) staging.
    "hier": Workload("hier", R=32, E=256, K=8, T=4096, H=7168, router="bias", bias_std=1.0,
                     num_nodes=4),
}


def _router(w: Workload, g: torch.Generator):
    n = w.R * w.T
    if w.router in ("normal", "bias"):
        logits = torch.randn(n, w.E, generator=g, dtype=torch.float32)
        if w.router == "bias":
            bias = torch.randn(w.E, generator=g, dtype=torch.float32) * w.bias_std
            logits = logits + bias
        vals, idx = torch.topk(logits, w.K, dim=1)
        weights = torch.softmax(vals, dim=1)
    elif w.router == "zipf":
        perm = torch.randperm(w.E, generator=g)
        ranks = torch.empty(w.E, dtype=torch.float64)
        ranks[perm] = torch.arange(1, w.E + 1, dtype=torch.float64)
        logp = (-w.zipf_s * torch.log(ranks)).to(torch.float32)
        u = torch.rand(n, w.E, generator=g, dtype=torch.float32).clamp_(1e-12, 1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        pert = logp.unsqueeze(0) + gumbel
        vals, idx = torch.topk(pert, w.K, dim=1)
        weights = torch.softmax(vals, dim=1)
    else:
        raise ValueError(f"unknown router {w.router!r}")
    idx = idx.to(torch.int64)
    if w.mask_p > 0.0:
        m = torch.rand(n, w.K, generator=g, dtype=torch.float32) < w.mask_p
        idx = torch.where(m, torch.full_like(idx, -1), idx)
    return idx.reshape(w.R, w.T, w.K).contiguous(), weights.to(torch.float32).reshape(w.R, w.T, w.K).contiguous()


def make_routing(w: Workload, seed: int = 0):
    """topk_idx [R][T][K] int64 and topk_weights [R][T][K] fp32 on the CPU."""
    g = torch.Generator().manual_seed(seed)
    return _router(w, g)


def make_x(w: Workload, seed: int = 0, device: Optional[str] = None) -> torch.Tensor:
    """x [R][T][H] bf16 ~ N(0, 1).

    Drawn on the CPU with a seeded generator unless ``device`` names a CUDA
    device, in which case a seeded CUDA generator draws it there (used for the
    largest workloads, where the CPU draw would dominate set-up time)."""
    if device is None or device == "cpu":
        g = torch.Generator().manual_seed(seed + 1)
        return torch.randn(w.R, w.T, w.H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    g = torch.Generator(device=device).manual_seed(seed + 1)
    out = torch.empty(w.R, w.T, w.H, dtype=torch.bfloat16, device=device)
    # draw in slabs to bound the fp32 temporary
    flat = out.view(-1, w.H)
    step = max(1, (1 << 26) // max(1, w.H))
    for i in range(0, flat.shape[0], step):
        j = min(flat.shape[0], i + step)
        flat[i:j] = torch.randn(j - i, w.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_inputs(w: Workload, seed: int = 0, x_device: Optional[str] = None):
    topk_idx, topk_weights = make_routing(w, seed)
    x = make_x(w, seed, x_device)
    return x, topk_idx, topk_weights


def random_topk(R: int, E: int, K: int, T: int, seed: int, mask_p: float = 0.0,
                distinct: bool = True) -> torch.Tensor:
    """Small random routings for property and edge-case tests."""
    g = torch.Generator().manual_seed(seed)
    if distinct:
        keys = torch.rand(R * T, E, generator=g)
        idx = torch.topk(keys, K, dim=1).indices.to(torch.int64)
    else:
        idx = torch.randint(0, E, (R * T, K), generator=g, dtype=torch.int64)
    if mask_p > 0:
        m = torch.rand(R * T, K, generator=g) < mask_p
        idx = torch.where(m, torch.full_like(idx, -1), idx)
    return idx.reshape(R, T, K).contiguous()


def random_weights(R: int, T: int, K: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed + 7)
    return torch.rand(R, T, K, generator=g, dtype=torch.float32)


def random_x(R: int, T: int, H: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed + 11)
    return torch.randn(R, T, H, generator=g, dtype=torch.float32).to(torch.bfloat16)


def random_rows(n: int, H: int, seed: int, device: Optional[str] = None) -> torch.Tensor:
    """[n][H] bf16: N(0, 1) values times a per-row power of two in 2^-4..2^4.

    A stand-in expert output with a different row for every permuted row or
    packed slot (unlike the identity expert, whose rows repeat the token's x
    for every k), so that a combine reading the wrong row of a token changes
    its result.  Drawn like ``make_x`` (CPU generator, or a seeded CUDA
    generator in slabs when ``device`` is a CUDA device)."""
    on_cpu = device is None or device == "cpu"
    g = torch.Generator(device="cpu" if on_cpu else device).manual_seed(seed + 23)
    dev = "cpu" if on_cpu else device
    out = torch.empty(n, H, dtype=torch.bfloat16, device=dev)
    step = max(1, (1 << 26) // max(1, H))
    for i in range(0, n, step):
        j = min(n, i + step)
        v = torch.randn(j - i, H, generator=g, device=dev, dtype=torch.float32)
        e = torch.randint(-4, 5, (j - i, 1), generator=g, device=dev).to(torch.float32)
        out[i:j] = (v * torch.exp2(e)).to(torch.bfloat16)
    return out
