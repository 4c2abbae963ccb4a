"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws Q, K, V (and the
upstream gradient dO for the backward).  The pages
measure on i.i.d. Gaussian tensors of shape (B, H, N, d) ("How to profile and
optimise kernels", section "How I profile": three torch.randn tensors viewed
as (B, H, N, D); the bench of "FlashAttention and kernels.", section "Build
It").  The heavy-tailed workload multiplies Q and K by 8 and replaces 1% of
their entries by +-40, to stress the running maximum and the rescaling.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple          # which masks this workload is run with
    values: str            # "normal" or "outliers"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("B1-H2-N256-d64", 1, 2, 256, 64, (False, True), "normal"),
        Workload("B4-H16-N1024-d64", 4, 16, 1024, 64, (False, True), "normal"),
        Workload("B1-H32-N4096-d128", 1, 32, 4096, 128, (False, True), "normal"),
        Workload("B1-H32-N32768-d128", 1, 32, 32768, 128, (True,), "normal"),
        Workload("B2-H8-N3001-d128-outliers", 2, 8, 3001, 128, (False, True), "outliers"),
    )
}

# the headline shape: N = 4096, d = 128
HEADLINE = "B1-H32-N4096-d128"


def make_qkv(B: int, H: int, N: int, d: int, seed: int = 0, values: str = "normal",
             device="cpu", dtype=torch.bfloat16):
    """Draw q, k, v of shape [B, H, N, d], contiguous, rounded to ``dtype``.

    values="normal": i.i.d. N(0, 1).
    values="outliers": q and k are N(0, 1) * 8, then 1% of their entries
    (a seeded Bernoulli mask) are set to +-40 with a random sign; v is N(0, 1).
    The draw is in float32 and rounded once to ``dtype``.
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (B, H, N, d)

    def normal():
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)

    q, k, v = normal(), normal(), normal()
    if values == "outliers":
        for t in (q, k):
            t.mul_(8.0)
            hit = torch.rand(shape, generator=g, device=device) < 0.01
            sign = torch.where(torch.rand(shape, generator=g, device=device) < 0.5, -1.0, 1.0)
            t.copy_(torch.where(hit, 40.0 * sign, t))
    elif values != "normal":
        raise ValueError(f"unknown value recipe {values!r}")
    return q.to(dtype).contiguous(), k.to(dtype).contiguous(), v.to(dtype).contiguous()


def make_grad(B: int, H: int, N: int, d: int, seed: int = 0, device="cpu", dtype=torch.bfloat16):
    """The upstream gradient dO for the backward: i.i.d. N(0, 1), [B, H, N, d], rounded to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 7919)
    return torch.randn((B, H, N, d), generator=g, device=device, dtype=torch.float32).to(dtype).contiguous()


def make_workload(name: str, seed: int = 0, device="cpu"):
    w = WORKLOADS[name]
    return make_qkv(w.B, w.H, w.N, w.d, seed=seed, values=w.values, device=device)
