"""Seeded synthetic inputs for causal GQA prefill.

This module holds no attention arithmetic. It draws the random q/k/v that
both the GPU library and the CPU oracle are given, so the two sides read the
very same bf16 bits.

The workloads stand in for the Qwen text-encoder prefill of antirez/h3.c
issue #47 (one concatenated multimodal sequence of video, image and prompt
tokens; the failing lengths 8184, 8199, 8510 and 10231 are from its
"Systematic single-variable experiments" table). There is no dataset or
checkpoint; the values are i.i.d. normal.

Recipe: numpy's PCG64 generator, `np.random.default_rng(seed)`, for the
outlier workload first `rng.permutation(D)[:n_outlier]` picks the channels
that are multiplied by 8 in q and k (all heads, all rows); then float64
standard normals are drawn in the order q [Hq,T,D], k [Hkv,T,D], v [Hkv,T,D]
(in slabs of rows; the stream is the same as one large draw); each value is
rounded to fp32 and to bf16 (round to nearest even). numpy's generator gives
the same stream on x86 and aarch64, so a given seed means the same bits on
every machine (torch's CPU randn does not: its vectorised math differs
between architectures in the last bit of a few values).
"""
from dataclasses import dataclass
from typing import Optional, Tuple

import numpy as np
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
    causal: bool = True         # False: every key of the sequence (bidirectional)

    @property
    def total_tokens(self) -> int:
        return sum(self.seqlens)

    @property
    def scale(self) -> float:
        return self.head_dim ** -0.5

    def metric_flops(self) -> float:
        """FLOPs as the headline metric counts them: sum_b 2*S_b^2*Hq*D
        (causal), 4*S_b^2*Hq*D without the causal rule."""
        k = 2.0 if self.causal else 4.0
        return float(sum(k * s * s * self.n_q_heads * self.head_dim for s in self.seqlens))

    def exact_flops(self) -> float:
        """FLOPs of the visible pairs: 4*D per (query, key, head) pair, i.e.
        2*Hq*D*S(S+1) per sequence when causal."""
        if not self.causal:
            return self.metric_flops()
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
    # Bidirectional attention at the DiT row counts of tgo-app-dev/vpipe
    # issue #10 (a 19316-row forward and a 34121-row forward), with the
    # encoder's head shape (a reading: the pages give no DiT head counts).
    "dit19316": Workload("dit19316", (19316,), seed=1006, causal=False),
    "dit34121": Workload("dit34121", (34121,), seed=1007, causal=False),
}

HEADLINE = "s10231"


def cu_seqlens_of(seqlens) -> torch.Tensor:
    cu = [0]
    for s in seqlens:
        cu.append(cu[-1] + int(s))
    return torch.tensor(cu, dtype=torch.int32)


def _normal_bf16(rng, shape, scale_channels=None, std=1.0):
    """Draws float64 normals row-slab by row-slab (bounded host memory) and
    returns the bf16 tensor. Channel scaling (x8) happens in fp32 before the
    bf16 rounding."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(-1, shape[-1])
    rows = flat.shape[0]
    step = max(1, (1 << 22) // shape[-1])
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        a = rng.standard_normal((r1 - r0, shape[-1])).astype(np.float32)
        if std != 1.0:
            a *= np.float32(std)
        if scale_channels is not None:
            a[:, scale_channels] *= np.float32(8.0)
        flat[r0:r1] = torch.from_numpy(a).to(torch.bfloat16)
    return out


def make_inputs(seqlens, n_q_heads: int, n_kv_heads: int, head_dim: int,
                seed: int, n_outlier: int = 0, std: float = 1.0):
    """Returns dict(q, k, v: bf16 CPU tensors; cu_seqlens: int32 CPU tensor;
    outlier_channels: the scaled channel indices, or None)."""
    T = sum(int(s) for s in seqlens)
    rng = np.random.default_rng(int(seed))
    idx = rng.permutation(head_dim)[:n_outlier] if n_outlier else None
    q = _normal_bf16(rng, (n_q_heads, T, head_dim), idx, std)
    k = _normal_bf16(rng, (n_kv_heads, T, head_dim), idx, std)
    v = _normal_bf16(rng, (n_kv_heads, T, head_dim), None, std)
    return {
        "q": q,
        "k": k,
        "v": v,
        "cu_seqlens": cu_seqlens_of(seqlens),
        "outlier_channels": None if idx is None else torch.from_numpy(np.asarray(idx)),
    }


def rope_tables(seqlens, head_dim: int, theta: float = 1.0e6):
    """Rotary tables [T, D/2] fp32 for positions counted from each sequence
    start: angle = pos * theta^(-2i/D), i < D/2 (the standard rotate-half
    frequencies; theta = 1e6 as in Qwen3 text models)."""
    half = head_dim // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / head_dim)
    pos = np.concatenate([np.arange(int(s), dtype=np.float64) for s in seqlens]) \
        if len(seqlens) else np.zeros(0)
    ang = pos[:, None] * inv[None, :]
    return (torch.from_numpy(np.cos(ang).astype(np.float32)),
            torch.from_numpy(np.sin(ang).astype(np.float32)))


def norm_weights(head_dim: int, seed: int):
    """Synthetic RMS-norm weights for q and k: 1 + 0.1 N(0,1), bf16 (there is no
    checkpoint); drawn from their own generator so the q/k/v draws are
    unchanged."""
    rng = np.random.default_rng(int(seed) + 7919)
    w = 1.0 + 0.1 * rng.standard_normal((2, head_dim))
    t = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16)
    return t[0].contiguous(), t[1].contiguous()


def make_workload_inputs(w: Workload):
    return make_inputs(w.seqlens, w.n_q_heads, w.n_kv_heads, w.head_dim,
                       w.seed, w.n_outlier)
