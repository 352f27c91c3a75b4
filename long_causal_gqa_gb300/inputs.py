"""Seeded synthetic inputs for causal GQA prefill.

This module holds no attention arithmetic. It draws the random q/k/v that
both the GPU library and the CPU oracle are given, so the two sides read the
very same bf16 bits.

The workloads stand in for the Qwen text-encoder prefill of antirez/h3.c
issue #47 (one concatenated multimodal sequence of video, image and prompt
tokens; the failing lengths 8184, 8199, 8510 and 10231 are from its
"Systematic single-variable experiments" table). There is no dataset or
checkpoint; the values are i.i.d. normal.

Recipe: fp32 `torch.randn` on the CPU from `torch.Generator().manual_seed(seed)`,
drawn in the order q [Hq,T,D], k [Hkv,T,D], v [Hkv,T,D]; for the outlier
workload, then `torch.randperm(D)[:n_outlier]` from the same generator picks
channels that are multiplied by 8 in q and k (all heads, all rows); finally
each tensor is rounded to bf16 (round to nearest even).
"""
from dataclasses import dataclass
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    seqlens: Tuple[int, ...]
    n_q_heads: int = 64
    n_kv_heads: int = 8
    head_dim: int = 128
    seed: int = 1000
    n_outlier: int = 0          # channels of q and k scaled by 8

    @property
    def total_tokens(self) -> int:
        return sum(self.seqlens)

    @property
    def scale(self) -> float:
        return self.head_dim ** -0.5

    def metric_flops(self) -> float:
        """FLOPs as the headline metric counts them: sum_b 2*S_b^2*Hq*D."""
        return float(sum(2.0 * s * s * self.n_q_heads * self.head_dim
                         for s in self.seqlens))

    def exact_flops(self) -> float:
        """FLOPs of the causal pairs actually needed: 2*Hq*D*S(S+1) per sequence
        (one QK^T and one PV multiply-add per visible (query, key) pair)."""
        return float(sum(2.0 * self.n_q_heads * self.head_dim * s * (s + 1)
                         for s in self.seqlens))


# The five measured workloads: S=512 (small, the oracle runs it in seconds),
# S=7700 (just under the ~7700-token capacity of the Metal kernel), S=10231
# (the failing length in the issue title; the headline workload), the four
# failing lengths packed as one varlen batch, and S=32768 with outlier
# channels. Seeds are 1000 + the workload's position (1..5).
WORKLOADS = {
    "s512": Workload("s512", (512,), seed=1001),
    "s7700": Workload("s7700", (7700,), seed=1002),
    "s10231": Workload("s10231", (10231,), seed=1003),
    "varlen4": Workload("varlen4", (8184, 8199, 8510, 10231), seed=1004),
    "s32768_outlier": Workload("s32768_outlier", (32768,), seed=1005, n_outlier=4),
}

HEADLINE = "s10231"


def cu_seqlens_of(seqlens) -> torch.Tensor:
    cu = [0]
    for s in seqlens:
        cu.append(cu[-1] + int(s))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(seqlens, n_q_heads: int, n_kv_heads: int, head_dim: int,
                seed: int, n_outlier: int = 0, std: float = 1.0):
    """Returns dict(q, k, v: bf16 CPU tensors; cu_seqlens: int32 CPU tensor;
    outlier_channels: the scaled channel indices, or None)."""
    T = sum(int(s) for s in seqlens)
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((n_q_heads, T, head_dim), generator=g, dtype=torch.float32)
    k = torch.randn((n_kv_heads, T, head_dim), generator=g, dtype=torch.float32)
    v = torch.randn((n_kv_heads, T, head_dim), generator=g, dtype=torch.float32)
    if std != 1.0:
        q.mul_(std)
        k.mul_(std)
        v.mul_(std)
    idx: Optional[torch.Tensor] = None
    if n_outlier:
        idx = torch.randperm(head_dim, generator=g)[:n_outlier]
        q[:, :, idx] *= 8.0
        k[:, :, idx] *= 8.0
    return {
        "q": q.to(torch.bfloat16),
        "k": k.to(torch.bfloat16),
        "v": v.to(torch.bfloat16),
        "cu_seqlens": cu_seqlens_of(seqlens),
        "outlier_channels": idx,
    }


def make_workload_inputs(w: Workload):
    return make_inputs(w.seqlens, w.n_q_heads, w.n_kv_heads, w.head_dim,
                       w.seed, w.n_outlier)
