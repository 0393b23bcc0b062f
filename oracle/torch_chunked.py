"""The page's chunked form in plain PyTorch CPU ops, fp32 -- a like-for-like CPU baseline.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: ``tests/`` pin it and the CPU-baseline
leg of ``bench.py`` times it; the CUDA path never imports it.

"Fractus-1B training optimization -- 2026-08-22", section 2, "Opt 2": inside a block of
tokens a masked block x block score matrix; across blocks the running state (S_run, z_run),
updated inclusively after the block has read it.  The page measures this form with PyTorch
on a CPU (section 4, "Measured results", the CPU micro-benchmark table: G = B * 40 groups,
128 tokens, head size 64, carry active, forward and forward + backward).  Here the same
steps, each a PyTorch operator, the backward by autograd -- the page's own way of running
it -- so that the GPU kernels can be set beside a CPU number of the same kind.

Reading (as for the whole oracle): o_t = q_t^T S_t / (q_t . z_t + eps) with S_t, z_t
inclusive of token t; S[p][c], p the key dimension.
"""
from __future__ import annotations

import torch


def chunked_fwd(q, k, v, S0=None, z0=None, block: int = 64, eps: float = 1e-6):
    """q, k, v: [G, C, D] fp32 CPU tensors; S0 [G, D, D], z0 [G, D] or None (zeros).
    Returns (o, S_out, z_out); differentiable."""
    G, C, D = q.shape
    S = torch.zeros(G, D, D, dtype=q.dtype) if S0 is None else S0
    z = torch.zeros(G, D, dtype=q.dtype) if z0 is None else z0
    outs = []
    for b0 in range(0, C, block):
        qb, kb, vb = q[:, b0:b0 + block], k[:, b0:b0 + block], v[:, b0:b0 + block]
        A = torch.tril(qb @ kb.transpose(1, 2))               # keys j <= t of the block
        num = qb @ S + A @ vb                                  # the state before the block, then the block
        den = (qb * z[:, None, :]).sum(-1) + A.sum(-1) + eps
        outs.append(num / den[..., None])
        S = S + kb.transpose(1, 2) @ vb                        # updated after the block read it
        z = z + kb.sum(1)
    return torch.cat(outs, 1), S, z


def chunked_fwd_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, block: int = 64, eps: float = 1e-6):
    """Forward, then autograd's backward for the upstream gradients (dO, dS_out, dz_out).
    Returns (o, S_out, z_out, dq, dk, dv, dS0, dz0)."""
    leaves = [t.detach().clone().requires_grad_(True) for t in (q, k, v, S0, z0)]
    o, S, z = chunked_fwd(*leaves, block=block, eps=eps)
    torch.autograd.backward((o, S, z), (dO, dS_out, dz_out))
    return (o.detach(), S.detach(), z.detach()) + tuple(t.grad for t in leaves)
