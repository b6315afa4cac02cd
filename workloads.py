"""Seeded synthetic workloads for exact attention.

This module only describes shapes and draws random inputs; it holds none of
the attention arithmetic. Both the CUDA path and the CPU oracle consume the
tensors it produces, so the two sides always see bit-identical bf16 values.

Recipe (one recipe for every workload):
  * a CPU ``torch.Generator`` seeded with ``seed``;
  * ``torch.randn`` in fp32, drawn in the order q, k, v, dO;
  * each tensor multiplied by its standard deviation (q and k share one);
  * rounded to bf16 with round-to-nearest-even (``Tensor.to(torch.bfloat16)``).

Layout is BSHD with the head dimension innermost: q, o, dO are
``[B, Nq, Hq, d]``; k, v are ``[B, Nk, Hkv, d]``.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    direction: str  # "fwd" or "bwd"
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self) -> float:
        """4*B*Hq*Nq*Nk*d, halved under the causal mask (the two GEMMs)."""
        f = 4.0 * self.B * self.Hq * self.Nq * self.Nk * self.d
        return f * 0.5 if self.causal else f

    def bwd_flops(self) -> float:
        """2.5x the forward count (five GEMMs against two)."""
        return 2.5 * self.fwd_flops()


# The five headline workloads (sizes, distributions and masks as published
# for the method's evaluation). Seeds are 1000 + position.
WORKLOADS = [
    Workload("fwd_b1_h2_n256_d64", "fwd", 1, 2, 2, 256, 256, 64, False, seed=1000),
    Workload("fwd_b4_h16_n2048_d128", "fwd", 4, 16, 16, 2048, 2048, 128, False, seed=1001),
    Workload("fwd_causal_b2_h16_n8192_d128", "fwd", 2, 16, 16, 8192, 8192, 128, True, seed=1002),
    Workload("fwd_causal_gqa_b1_hq32_hkv8_n16384_d128", "fwd", 1, 32, 8, 16384, 16384, 128, True,
             sigma_qk=2.0, seed=1003),
    Workload("bwd_causal_b4_h16_n4096_d128", "bwd", 4, 16, 16, 4096, 4096, 128, True, seed=1004),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def make_inputs(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, seed: int,
                sigma_qk: float = 1.0, sigma_v: float = 1.0, with_dout: bool = False,
                sigma_do: float = 1.0) -> dict:
    """Draw q, k, v (and dO) as CPU bf16 tensors in BSHD layout."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    out["q"] = (torch.randn((B, Nq, Hq, d), generator=g, dtype=torch.float32) * sigma_qk).to(torch.bfloat16)
    out["k"] = (torch.randn((B, Nk, Hkv, d), generator=g, dtype=torch.float32) * sigma_qk).to(torch.bfloat16)
    out["v"] = (torch.randn((B, Nk, Hkv, d), generator=g, dtype=torch.float32) * sigma_v).to(torch.bfloat16)
    if with_dout:
        out["do"] = (torch.randn((B, Nq, Hq, d), generator=g, dtype=torch.float32) * sigma_do).to(torch.bfloat16)
    return out


def workload_inputs(w: Workload, with_dout: bool | None = None) -> dict:
    if with_dout is None:
        with_dout = w.direction == "bwd"
    return make_inputs(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.seed, w.sigma_qk, w.sigma_v, with_dout)
