"""Seeded synthetic inputs for the fused GEMM + scale + ReLU operator.

This module only draws numbers; it holds none of the operator's arithmetic, so
the GPU parity tests, the benchmark and the CPU oracle can all take their
inputs from it without sharing any of the method.

Recipe (page "Tutorial14: 使用TileLang语言编写attention算子", section 2, the
main() of the tutorial script): seed the CPU generator, draw A = randn(M, K) in
float32 and round it to float16, then draw B = randn(K, N) the same way, A
first.  The LLM-shaped and skinny workloads draw B with standard deviation
1/sqrt(K) (B = randn * K**-0.5 before the rounding), as a trained projection
matrix would have.  The pages use no public dataset; these stand in for it.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    b_std_inv_sqrt_k: bool = False   # B ~ N(0, 1/K) instead of N(0, 1)
    note: str = ""

    @property
    def flops(self) -> int:
        """Algorithmic work: one multiply and one add per (m, n, k)."""
        return 2 * self.M * self.N * self.K

    @property
    def bytes(self) -> int:
        """Algorithmic HBM traffic: A and B read once, C written once (fp16)."""
        return 2 * (self.M * self.K + self.K * self.N + self.M * self.N)


# The five workloads the library is measured and checked on.
WORKLOADS = {
    "square1024": Workload("square1024", 1024, 1024, 1024, 0.5,
                           note="the tutorial's own instance"),
    "ragged2000x3000x1000": Workload("ragged2000x3000x1000", 2000, 3000, 1000, 1.0,
                                     note="tile-edge predication and masking"),
    "square8192": Workload("square8192", 8192, 8192, 8192, 0.5,
                           note="tensor-core-bound steady state"),
    "llm_mlp_up": Workload("llm_mlp_up", 16384, 14336, 4096, 1.0, True,
                           note="LLM MLP up-projection: 16384 tokens, K=4096, N=14336"),
    "skinny_decode": Workload("skinny_decode", 16, 16384, 16384, 0.5, True,
                              note="decode-like skinny shape, HBM-bound"),
}


def make_inputs(M: int, N: int, K: int, seed: int = 0, b_std_inv_sqrt_k: bool = False):
    """Return (A, B) as contiguous float16 CPU tensors drawn from ``seed``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    A = torch.randn(M, K, generator=g, dtype=torch.float32).half()
    B = torch.randn(K, N, generator=g, dtype=torch.float32)
    if b_std_inv_sqrt_k and K > 0:
        B = B * (float(K) ** -0.5)
    B = B.half()
    return A.contiguous(), B.contiguous()


def workload_inputs(w: Workload, seed: int = 0):
    return make_inputs(w.M, w.N, w.K, seed=seed, b_std_inv_sqrt_k=w.b_std_inv_sqrt_k)


def sample_rows(M: int, count: int = 128, seed: int = 1234):
    """Seeded sample of whole output rows: ``count`` random rows plus the tile edges
    {0, 127, 128, M-1} (those that exist), sorted and unique."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    n = min(count, M)
    picked = torch.randperm(M, generator=g)[:n].tolist() if M > 0 else []
    edges = [r for r in (0, 127, 128, M - 1) if 0 <= r < M]
    return sorted(set(picked) | set(edges))


def make_bias(N: int, seed: int = 0):
    """Seeded bias vector for the bias + GELU epilogue: randn(N) * 2 rounded to fp16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (torch.randn(N, generator=g, dtype=torch.float32) * 2).half().contiguous()


@dataclass(frozen=True)
class AttnWorkload:
    """Attention forward: Q (B,H,S,D), K/V (B,H,S,D), fp16, randn inputs."""
    name: str
    B: int
    H: int
    S: int
    D: int
    causal: bool

    @property
    def pairs(self) -> int:
        """(query, key) pairs that are not masked, per head."""
        return self.S * (self.S + 1) // 2 if self.causal else self.S * self.S

    @property
    def flops(self) -> int:
        """Q K^T and P V: 2 x 2 D flops per unmasked (query, key) pair."""
        return 4 * self.B * self.H * self.D * self.pairs


ATTN_WORKLOADS = {
    w.name: w for w in (
        AttnWorkload("attn_b4_h32_s4096_d128", 4, 32, 4096, 128, False),
        AttnWorkload("attn_b4_h32_s4096_d128_causal", 4, 32, 4096, 128, True),
        AttnWorkload("attn_b8_h16_s2048_d64", 8, 16, 2048, 64, False),
    )
}


def attention_inputs(w: AttnWorkload, seed: int = 0, device="cpu"):
    """Q, K, V float16 from randn (drawn on ``device`` with a seeded generator)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (w.B, w.H, w.S, w.D)
    return tuple(torch.randn(shape, generator=g, device=device, dtype=torch.float32).half()
                 for _ in range(3))
