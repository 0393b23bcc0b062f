"""Seeded synthetic inputs for chunked causal linear attention.

This module only draws random numbers and rounds them to the requested dtype.  It
holds none of the method's arithmetic and is the one piece of code that both the
CUDA path's tests/bench and the fp64 oracle consume: the same bits go to both.

Distributions (the workloads of the Fractus-1B attention micro-benchmark, G groups
of C tokens with head size D, carry active):

* q, k = softplus(N(0, 1))  -- positive features, so every denominator is > 0
* v ~ N(0, 1)
* S0 = sum of m = 32 outer products k'_m v'_m^T, z0 = sum_m k'_m, with
  k' = softplus(N(0, 1)) and v' ~ N(0, 1)   (a carry that looks like 32 earlier tokens)
* upstream gradients: dO ~ N(0, 1); dS_out, dz_out ~ N(0, 0.01^2) (0.01 read as the
  standard deviation)

Everything is drawn in float32 on the CPU from ``torch.Generator().manual_seed(seed)``
in a fixed order, then q, k, v, dO are rounded to the compute dtype.  Carries and
carry gradients stay float32.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

CARRY_TERMS = 32


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    S0: Optional[torch.Tensor]
    z0: Optional[torch.Tensor]
    dO: Optional[torch.Tensor] = None
    dS_out: Optional[torch.Tensor] = None
    dz_out: Optional[torch.Tensor] = None

    def tensors(self):
        return {k: v for k, v in self.__dict__.items() if v is not None}

    def to(self, device) -> "Inputs":
        return Inputs(**{k: (None if v is None else v.to(device)) for k, v in self.__dict__.items()})


def _dtype(name) -> torch.dtype:
    if isinstance(name, torch.dtype):
        return name
    return {"bf16": torch.bfloat16, "bfloat16": torch.bfloat16,
            "f32": torch.float32, "fp32": torch.float32, "float32": torch.float32}[name]


def make_inputs(G: int, C: int, D: int, dtype="bf16", seed: int = 0, carry: bool = True,
                grads: bool = False, carry_terms: int = CARRY_TERMS) -> Inputs:
    """Draw one workload.  ``carry=False`` leaves S0/z0 as None (zero carry);
    ``grads=True`` also draws dO, dS_out, dz_out."""
    dt = _dtype(dtype)
    gen = torch.Generator().manual_seed(int(seed))
    sp = torch.nn.functional.softplus
    q = sp(torch.randn(G, C, D, generator=gen))
    k = sp(torch.randn(G, C, D, generator=gen))
    v = torch.randn(G, C, D, generator=gen)
    S0 = z0 = None
    if carry:
        kp = sp(torch.randn(G, carry_terms, D, generator=gen))
        vp = torch.randn(G, carry_terms, D, generator=gen)
        S0 = torch.bmm(kp.transpose(1, 2), vp).contiguous()
        z0 = kp.sum(dim=1).contiguous()
    dO = dS_out = dz_out = None
    if grads:
        dO = torch.randn(G, C, D, generator=gen).to(dt).contiguous()
        dS_out = (0.01 * torch.randn(G, D, D, generator=gen)).contiguous()
        dz_out = (0.01 * torch.randn(G, D, generator=gen)).contiguous()
    return Inputs(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                  S0=S0, z0=z0, dO=dO, dS_out=dS_out, dz_out=dz_out)


# The five workloads the implementation is checked and measured on.
CONFIGS = {
    "tiny_f32": dict(G=8, C=128, D=64, block=64, dtype="f32", eps=1e-6),
    "fractus1b_fwd": dict(G=160, C=128, D=64, block=64, dtype="bf16", eps=1e-6),
    "fractus1b_fwdbwd_b16": dict(G=640, C=128, D=64, block=64, dtype="bf16", eps=1e-6),
    "long_stream": dict(G=160, C=128, D=64, block=64, dtype="bf16", eps=1e-6, chunks=64),
    "wide_d128": dict(G=320, C=256, D=128, block=64, dtype="bf16", eps=1e-6),
}


# The tied head of the Fractus-1B model: d_model 1280 (64.3M MACs per token over a
# 50257-token vocabulary), 512 tokens per training tick (B = 4 sequences of 128).
CE_SHAPE = dict(N=512, V=50257, d=1280)


def make_ce_inputs(N: int, V: int, d: int, seed: int = 0):
    """Hidden rows h ~ N(0, 1) and a head W ~ N(0, 0.02^2), both rounded to bfloat16,
    and targets uniform in [0, V) (int32).  Logits h . W_j then have a standard deviation
    near 0.02 sqrt(d) (0.7 at d = 1280).  Returns (h, W, targets) on the CPU."""
    gen = torch.Generator().manual_seed(int(seed))
    h = torch.randn(N, d, generator=gen).to(torch.bfloat16).contiguous()
    W = (0.02 * torch.randn(V, d, generator=gen)).to(torch.bfloat16).contiguous()
    y = torch.randint(0, V, (N,), generator=gen, dtype=torch.int64).to(torch.int32).contiguous()
    return h, W, y
