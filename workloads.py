"""Seeded synthetic workloads.

Shapes, dtypes and degrees of the workloads, and the seeded generator of
their inputs.  This module holds none of the attention arithmetic and imports
neither the library nor the oracle: it is the one piece that both the CUDA
path (through the tests and the benchmark) and the CPU oracle are fed from.

Input recipe: ``torch.Generator('cpu').manual_seed(seed)`` (seed 0 by
default), then ``q, k, v = randn(shape, float32)`` drawn in that order, then a
round-to-nearest-even cast to the workload dtype.  Values are N(0, 1) with no
structure, standing in for the FLUX.1-dev and video-model activations that the
Diffusers "Context parallelism" guide and the ParaAttention README benchmark
(no dataset or weights are used).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    seq: int
    head_dim: int
    dtype: str               # "f32" or "bf16"
    ring_degree: int = 1
    ring_anything: bool = False
    ulysses_degree: int = 1
    layout: str = "bhsd"     # "bhsd": [B, H, S, D]; "bshd": [B, S, H, D]
    description: str = ""
    causal: bool = False     # query i attends keys j <= i
    ulysses_anything: bool = False   # uneven head groups (tensor_split sizes)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def shape(self):
        if self.layout == "bshd":
            return (self.batch, self.seq, self.heads, self.head_dim)
        return (self.batch, self.heads, self.seq, self.head_dim)

    @property
    def flops(self) -> float:
        """4 * B * H * D * (query, key) pairs: Q K^T plus P V, exp not
        counted, no padding counted; S^2 pairs, or S (S + 1) / 2 causal."""
        pairs = self.seq * (self.seq + 1) / 2 if self.causal else self.seq * self.seq
        return 4.0 * self.batch * self.heads * pairs * self.head_dim


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_ring", 1, 2, 256, 64, "f32", ring_degree=4,
                 description="tiny ring: fp32 [1,2,256,64], ring_degree 4"),
        Workload("flux_ring", 1, 24, 4608, 128, "bf16", ring_degree=2,
                 description="FLUX-like joint attention (4096 image + 512 text "
                             "tokens): bf16 [1,24,4608,128], ring_degree 2"),
        Workload("ulysses", 1, 24, 4608, 128, "bf16", ulysses_degree=4, layout="bshd",
                 description="Ulysses regroup + attention: bf16 [1,4608,24,128] "
                             "(B,S,H,D), ulysses_degree 4"),
        Workload("video_ring", 1, 24, 32768, 128, "bf16", ring_degree=8,
                 description="video-like long sequence: bf16 [1,24,32768,128], "
                             "ring_degree 8"),
        Workload("uneven_ring", 2, 24, 4609, 128, "bf16", ring_degree=3, ring_anything=True,
                 description="ring_anything uneven split: bf16 [2,24,4609,128], "
                             "ring_degree 3"),
        Workload("flux_ring_causal", 1, 24, 4608, 128, "bf16", ring_degree=2, causal=True,
                 description="FLUX-like shape with causal masking: bf16 [1,24,4608,128], "
                             "ring_degree 2, is_causal"),
        Workload("unified", 1, 24, 4608, 128, "bf16", ring_degree=2, ulysses_degree=2,
                 layout="bshd",
                 description="Unified (Ulysses x Ring) on the FLUX-like shape: bf16 "
                             "[1,4608,24,128] (B,S,H,D), ulysses_degree 2, ring_degree 2"),
        Workload("ulysses_anything", 1, 24, 4608, 128, "bf16", ulysses_degree=5,
                 ulysses_anything=True, layout="bshd",
                 description="Ulysses Anything on the FLUX-like shape: bf16 [1,4608,24,128] "
                             "(B,S,H,D), ulysses_degree 5 (24 heads -> 5 5 5 5 4; "
                             "4608 tokens not divisible by 5)"),
    ]
}


def make_qkv(shape, dtype: torch.dtype, seed: int = 0,
             device: Optional[str] = None):
    """q, k, v ~ N(0, 1) from one CPU generator, drawn in that order in fp32,
    then cast (RNE) to ``dtype``; optionally moved to ``device``."""
    g = torch.Generator("cpu").manual_seed(seed)
    out = []
    for _ in range(3):
        t = torch.randn(shape, dtype=torch.float32, generator=g).to(dtype)
        out.append(t.to(device) if device is not None else t)
    return tuple(out)


def make_workload(name: str, seed: int = 0, device: Optional[str] = None):
    w = WORKLOADS[name]
    return (w,) + make_qkv(w.shape, w.torch_dtype, seed, device)


def make_partials(rows_shape, head_dim: int, seed: int = 0, lse_spread: float = 4.0):
    """Two synthetic fp32 partials (out_a, lse_a, out_b, lse_b) for merge
    workloads: outputs ~ N(0, 1), LSEs ~ N(0, lse_spread^2) + 8."""
    g = torch.Generator("cpu").manual_seed(seed)
    o_a = torch.randn(*rows_shape, head_dim, generator=g)
    o_b = torch.randn(*rows_shape, head_dim, generator=g)
    l_a = torch.randn(*rows_shape, generator=g) * lse_spread + 8.0
    l_b = torch.randn(*rows_shape, generator=g) * lse_spread + 8.0
    return o_a, l_a, o_b, l_b
