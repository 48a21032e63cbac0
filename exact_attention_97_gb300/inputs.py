"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws i.i.d. N(0, 1)
tensors from a CPU ``torch.Generator`` and names the workloads. Both the CUDA
path and the CPU oracle receive exactly these values (bf16 values upcast
exactly to fp64 on the oracle side).

Seed convention for a workload seeded ``s``: Q from s, K from s+1, V from
s+2 and the upstream gradient dO from s+3. Values are drawn in fp32 and then
rounded to the workload's dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str  # "bf16" or "f32"
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int = 0
    Nk: int = 0  # key/value rows per head; 0 means N (the square problem)

    @property
    def n_keys(self) -> int:
        return self.Nk or self.N

    def pairs_per_head(self) -> float:
        """(query, key) pairs inside the mask: Nq*Nk, or under the causal mask
        aligned bottom-right (query i sees keys j <= i + Nk - Nq) the sum of
        min(Nk, i + 1 + Nk - Nq) over the Nq queries."""
        nq, nk = self.N, self.n_keys
        if not self.causal:
            return float(nq) * nk
        off = nk - nq
        return float(nq) * off + nq * (nq + 1) / 2.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def flops_fwd(self) -> float:
        """4*d per (query, key) pair in the mask (two contractions): 4*B*H*N^2*d for
        the square problem, halved under the causal mask (the N/2 diagonal term of
        the exact pair count is dropped, as in the usual convention)."""
        if self.n_keys == self.N:
            f = 4.0 * self.B * self.H * self.N * self.N * self.d
            return f / 2 if self.causal else f
        return 4.0 * self.B * self.H * self.d * self.pairs_per_head()

    def flops_bwd(self) -> float:
        """2.5x the forward count (five contractions instead of two)."""
        return 2.5 * self.flops_fwd()


# The five workloads of the method's evaluation, named by what they are.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("f32_B1_H2_N256_d64", "f32", 1, 2, 256, 64, False),
        Workload("bf16_causal_B1_H8_N1024_d64", "bf16", 1, 8, 1024, 64, True),
        Workload("bf16_B4_H16_N4096_d64", "bf16", 4, 16, 4096, 64, False),
        Workload("bf16_B8_H32_N4096_d128", "bf16", 8, 32, 4096, 128, False),
        Workload("bf16_causal_B1_H32_N65536_d128", "bf16", 1, 32, 65536, 128, True),
    ]
}

HEADLINE = "bf16_B8_H32_N4096_d128"


def randn(shape, seed: int, dtype=torch.float32) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(dtype)


def make_qkv_do(B: int, H: int, N: int, d: int, seed: int = 0, dtype=torch.bfloat16):
    """Host tensors (Q, K, V, dO), each [B, H, N, d], contiguous."""
    shape = (B, H, N, d)
    return tuple(randn(shape, seed + t, dtype) for t in range(4))


def workload_inputs(w: Workload):
    return make_qkv_do(w.B, w.H, w.N, w.d, w.seed, w.torch_dtype)


def sample_indices(n: int, count: int, seed: int) -> torch.Tensor:
    """``count`` distinct sorted indices in [0, n), seeded."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    count = min(count, n)
    return torch.randperm(n, generator=g)[:count].sort().values
