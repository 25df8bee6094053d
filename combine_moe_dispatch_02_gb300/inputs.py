"""Seeded synthetic inputs for MoE dispatch / combine.

This module holds no arithmetic of the operators: it draws token activations,
router logits and expert outputs, and turns the logits into a top-K routing
(the router itself is an input to dispatch, not part of it).  Both the CUDA
path and the CPU oracle are fed from here, so neither depends on the other.

Workloads (shapes follow the pages' examples):
  * tiny       -- 256 tokens, hidden 128, 16 experts / 4 ranks, top-2
  * dsv3       -- DeepSeek-V3 shape: 4096 tokens/rank, hidden 7168, 256 experts
                  over 8 ranks, top-8 ("MoE / Hybrid-EP Validation", measured-
                  reference table; Hybrid-EP news article, "Why This Issues
                  for AI Infrastructure": 8 of 256 experts per token)
  * dsv3_fp8   -- same routing, FP8 E4M3 dispatch
  * qwen_skew  -- Qwen3-235B-like: 8192 tokens, hidden 4096, 128 experts over
                  8 ranks, top-8, router logits biased by -1.2 * ln(e + 1)
                  (Zipf s = 1.2 popularity in expert-id order)
  * ds16_wide  -- DeepSeek-16B-like wide EP: 16384 tokens, hidden 2048, 64
                  experts over 32 ranks, top-6 ("Inside the Nebius + PyTorch
                  DeepSeek V3 recipe", "Benchmarking DeepEP on Nebius")

Recipe (torch CPU generator, ``torch.manual_seed(seed)``, drawn in this
order): x ~ N(0,1) fp32 [T,H] rounded to bf16; logits ~ N(0,1) fp32 [T,E]
(plus the Zipf bias for qwen_skew); probabilities = softmax(logits); top-K by
a stable descending sort (equal probabilities -> lower expert id first);
weights = top-K probabilities renormalised to sum to 1 in fp32; then, only if
asked for, y ~ N(0,1) fp32 [T*K,H] rounded to bf16 (expert outputs in the
expert-major row order).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    H: int          # hidden size
    E: int          # experts
    R: int          # virtual EP ranks
    K: int          # top-k
    fp8: bool = False
    zipf_s: float = 0.0

    @property
    def capacity(self) -> int:
        """Worst-case number of (token, rank) pairs: T * min(K, R)."""
        return self.T * min(self.K, self.R)

    def scaled(self, T: int) -> "Workload":
        return replace(self, name=f"{self.name}@T{T}", T=T)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 128, 16, 4, 2),
    "dsv3": Workload("dsv3", 4096, 7168, 256, 8, 8),
    "dsv3_fp8": Workload("dsv3_fp8", 4096, 7168, 256, 8, 8, fp8=True),
    "qwen_skew": Workload("qwen_skew", 8192, 4096, 128, 8, 8, zipf_s=1.2),
    "ds16_wide": Workload("ds16_wide", 16384, 2048, 64, 32, 6),
}


@dataclass
class Inputs:
    wl: Workload
    x: torch.Tensor          # bf16 [T,H]
    topk_idx: torch.Tensor   # int32 [T,K]
    topk_w: torch.Tensor     # fp32 [T,K]
    y: torch.Tensor | None   # bf16 [T*K,H] or None


def route(logits: torch.Tensor, K: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Top-K routing from router logits: stable descending sort of the softmax
    probabilities, weights renormalised over the chosen K (all fp32)."""
    probs = torch.softmax(logits.float(), dim=-1)
    vals, idx = torch.sort(probs, dim=-1, descending=True, stable=True)
    vals, idx = vals[:, :K].contiguous(), idx[:, :K].contiguous()
    w = vals / vals.sum(dim=-1, keepdim=True)
    return idx.to(torch.int32), w.float().contiguous()


def make_inputs(wl: Workload, seed: int = 0, with_y: bool = True) -> Inputs:
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(wl.T, wl.H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    logits = torch.randn(wl.T, wl.E, generator=g, dtype=torch.float32)
    if wl.zipf_s:
        bias = torch.tensor([-wl.zipf_s * math.log(e + 1.0) for e in range(wl.E)], dtype=torch.float32)
        logits = logits + bias
    idx, w = route(logits, wl.K)
    y = None
    if with_y:
        y = torch.randn(wl.T * wl.K, wl.H, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return Inputs(wl, x.contiguous(), idx, w, y)


def random_routing(T: int, K: int, E: int, seed: int, mask_frac: float = 0.0,
                   allow_duplicates: bool = False) -> torch.Tensor:
    """Uniform random expert ids for edge-case tests: distinct per row unless
    ``allow_duplicates``; a fraction of entries replaced by -1 (masked)."""
    g = torch.Generator().manual_seed(seed)
    if allow_duplicates:
        idx = torch.randint(0, E, (T, K), generator=g, dtype=torch.int64)
    else:
        idx = torch.argsort(torch.rand(T, E, generator=g), dim=-1)[:, :K]
    if mask_frac > 0:
        m = torch.rand(T, K, generator=g) < mask_frac
        idx = torch.where(m, torch.full_like(idx, -1), idx)
    return idx.to(torch.int32).contiguous()


def random_weights(T: int, K: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed + 7919)
    w = torch.rand(T, K, generator=g, dtype=torch.float32) + 0.05
    return (w / w.sum(dim=-1, keepdim=True)).contiguous()


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (a view, no arithmetic)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
