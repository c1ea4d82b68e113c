"""Seeded synthetic workloads for the attention forward pass.

This module only draws inputs; it holds none of the attention arithmetic, so
both the CUDA path's tests and the oracle's tests take their inputs from here.

The pages time and test attention on ``torch.randn`` tensors of shape
[B, H, N, d] ("4.4 Writing GPU Kernels with Triton", Kernel 4 self-check;
"Triton Kernel Practice", the FlashAttention core call). The five workloads
below follow that recipe at the sizes this library is measured on:

* a CPU ``torch.Generator`` seeded once per workload,
* ``torch.randn(B, H, N, d, dtype=float32)`` drawn for Q, then K, then V,
* each cast to bf16 (round to nearest even),
* Q and K then multiplied by ``logit_mult`` (a power of two, so exact in bf16).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    logit_mult: float = 1.0

    @property
    def scale(self) -> float:
        """1/sqrt(d), rounded to the fp32 value that crosses the C ABI."""
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def flops(self) -> float:
        """Counted FLOPs: 4*B*H*N^2*d, half of that under causal masking."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def describe(self) -> str:
        c = "causal" if self.causal else "non-causal"
        extra = f", Q,K x{self.logit_mult:g}" if self.logit_mult != 1.0 else ""
        return (f"attention fwd {c} B={self.B} H={self.H} N={self.N} d={self.d}"
                f" bf16 N(0,1){extra}")


# The five measured workloads (seed = position, 1-based).
SMALL = Workload("small_b1h2n256d64", 1, 2, 256, 64, False, 1)
MEDIUM = Workload("b4h16n1024d64", 4, 16, 1024, 64, False, 2)
CAUSAL_2K = Workload("causal_b4h16n2048d128", 4, 16, 2048, 128, True, 3)
CAUSAL_8K = Workload("causal_b2h16n8192d128", 2, 16, 8192, 128, True, 4)
TAIL_4000 = Workload("tail_b8h32n4000d64_x4", 8, 32, 4000, 64, False, 5, 4.0)

WORKLOADS = (SMALL, MEDIUM, CAUSAL_2K, CAUSAL_8K, TAIL_4000)

# Wider head dims (the page's d = 64 / 128 examples extended to 256 by the same
# zero-padding reading), measured beside the five above.
CAUSAL_4K_D256 = Workload("causal_b2h16n4096d256", 2, 16, 4096, 256, True, 6)
WIDE_2K_D256 = Workload("b4h16n2048d256", 4, 16, 2048, 256, False, 7)
EXTRA_WORKLOADS = (CAUSAL_4K_D256, WIDE_2K_D256)

BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}


def make_qkv(B: int, H: int, N: int, d: int, seed: int, logit_mult: float = 1.0, dtype=torch.bfloat16):
    """Seeded Q, K, V on the CPU, contiguous [B, H, N, d], bf16 (or ``dtype``, e.g. fp16)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = []
    for _ in range(3):
        x = torch.randn((B, H, N, d), dtype=torch.float32, generator=g)
        out.append(x.to(dtype))
    q, k, v = out
    if logit_mult != 1.0:
        q = q * logit_mult
        k = k * logit_mult
    return q.contiguous(), k.contiguous(), v.contiguous()


def workload_qkv(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.logit_mult)
