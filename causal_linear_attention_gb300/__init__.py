"""Chunked causal linear attention with a carried running state, for GB300 (sm_103a).

Per group g (G = B * levels * heads independent problems) and token t, with
S_t = S0 + sum_{j<=t} k_j v_j^T and z_t = z0 + sum_{j<=t} k_j (inclusive of t):

    o_t = (q_t^T S_t) / (q_t . z_t + eps),    final carry (S_{C-1}, z_{C-1})

("Fractus-1B training optimization -- 2026-08-22", section 2 "Opt 2": a masked
block x block score matrix inside a block plus the running state across blocks;
backward = the reverse cumsum of section 1.)  The kernels live in libla.so behind
the C ABI of include/la.h; this package only marshals arguments.

    import causal_linear_attention_gb300 as la
    o, S, z = la.chunked_fwd(q, k, v, S0, z0, block=64)          # q, k, v: [G, C, D] cuda
    dq, dk, dv, dS0, dz0 = la.chunked_bwd(q, k, v, S0, z0, dO, dS, dz, block=64)
"""
from __future__ import annotations

from typing import Optional

from ._lib import (LA_BF16, LA_F32, LAError, build, la_bwd_max_c, la_bwd_split_workspace_bytes, la_chunked_bwd,
                   la_chunked_bwd_split, la_chunked_fwd, la_chunked_fwd_split, la_chunked_fwd_split_static,
                   la_ce_bwd, la_ce_fwd, la_ce_workspace_bytes, la_chunked_step_host, la_cumsum_bwd,
                   la_cumsum_bwd_workspace_bytes, la_cumsum_fwd,
                   la_device_status, la_fwd_split_workspace_bytes, la_host_copy_eligible,
                   la_selftest_bounded_wait, la_status_string, la_step_workspace_bytes, la_version, lib)

__all__ = ["chunked_fwd", "chunked_fwd_split", "chunked_bwd", "chunked_bwd_split", "chunked_step_host",
           "step_workspace", "la_chunked_fwd", "la_chunked_fwd_split", "la_chunked_fwd_split_static",
           "la_fwd_split_workspace_bytes", "la_chunked_bwd", "la_chunked_bwd_split", "la_bwd_split_workspace_bytes",
           "cumsum_fwd", "cumsum_bwd", "la_cumsum_fwd", "la_cumsum_bwd", "la_cumsum_bwd_workspace_bytes",
           "ce_workspace", "ce_fwd", "ce_bwd", "la_ce_workspace_bytes", "la_ce_fwd", "la_ce_bwd",
           "la_chunked_step_host", "la_step_workspace_bytes", "la_host_copy_eligible", "la_bwd_max_c",
           "la_device_status",
           "la_selftest_bounded_wait",
           "la_status_string", "la_version", "build", "lib", "LAError", "LA_F32", "LA_BF16"]


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return LA_BF16
    if t.dtype == torch.float32:
        return LA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_tensor(name, t, shape, dtype, device):
    if t.shape != shape or t.dtype != dtype or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {tuple(shape)} {dtype} on {device}, "
                         f"got {tuple(t.shape)} {t.dtype} on {t.device} (contiguous={t.is_contiguous()})")


def chunked_fwd(q, k, v, S0=None, z0=None, *, block: int = 64, eps: float = 1e-6,
                o=None, S_out=None, z_out=None, stream=None):
    """Forward of one chunk.  q, k, v: contiguous [G, C, D] bf16 or fp32 CUDA tensors;
    S0 [G, D, D], z0 [G, D] fp32 or None (zero carry).  Returns (o, S_out, z_out);
    pass S_out=S0, z_out=z0 to thread the carry in place."""
    import torch
    G, C, D = q.shape
    dt = q.dtype
    for n, t in (("k", k), ("v", v)):
        _check_tensor(n, t, q.shape, dt, q.device)
    _check_tensor("q", q, q.shape, dt, q.device)
    for n, t, shp in (("S0", S0, (G, D, D)), ("z0", z0, (G, D))):
        if t is not None:
            _check_tensor(n, t, torch.Size(shp), torch.float32, q.device)
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(G, D, D, device=q.device, dtype=torch.float32) if S_out is None else S_out
    z_out = torch.empty(G, D, device=q.device, dtype=torch.float32) if z_out is None else z_out
    la_chunked_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, block, _dtype_code(q), eps, _stream(stream))
    return o, S_out, z_out


def chunked_fwd_split(q, k, v, S0=None, z0=None, *, block: int = 64, eps: float = 1e-6, o=None, S_out=None,
                      z_out=None, workspace=None, stream=None):
    """chunked_fwd cut along the tokens for few groups of long chunks (bf16, D = 64 or 128): the
    pieces of every group run on separate CTAs from carries computed by a prefix over the
    pieces' own sums.  `workspace` (a CUDA tensor of at least la_fwd_split_workspace_bytes
    bytes) is allocated here when not given.  Returns (o, S_out, z_out)."""
    import torch
    G, C, D = q.shape
    dt = q.dtype
    for n, t in (("k", k), ("v", v)):
        _check_tensor(n, t, q.shape, dt, q.device)
    _check_tensor("q", q, q.shape, dt, q.device)
    for n, t, shp in (("S0", S0, (G, D, D)), ("z0", z0, (G, D))):
        if t is not None:
            _check_tensor(n, t, torch.Size(shp), torch.float32, q.device)
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(G, D, D, device=q.device, dtype=torch.float32) if S_out is None else S_out
    z_out = torch.empty(G, D, device=q.device, dtype=torch.float32) if z_out is None else z_out
    need = la_fwd_split_workspace_bytes(G, C, D, _dtype_code(q))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    la_chunked_fwd_split(q, k, v, S0, z0, o, S_out, z_out, G, C, D, block, _dtype_code(q), eps, workspace, wbytes,
                         _stream(stream))
    return o, S_out, z_out


def _bwd_args(q, k, v, S0, z0, dO, dS_out, dz_out, out):
    import torch
    G, C, D = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _check_tensor(n, t, q.shape, q.dtype, q.device)
    for n, t, shp in (("S0", S0, (G, D, D)), ("z0", z0, (G, D)), ("dS_out", dS_out, (G, D, D)),
                      ("dz_out", dz_out, (G, D))):
        if t is not None:
            _check_tensor(n, t, torch.Size(shp), torch.float32, q.device)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q),
               torch.empty(G, D, D, device=q.device, dtype=torch.float32),
               torch.empty(G, D, device=q.device, dtype=torch.float32))
    return out


def ce_workspace(N: int, V: int, d: int, ce_chunk: int, device=None):
    """Device workspace (uint8 CUDA tensor) for ce_fwd / ce_bwd on this shape."""
    import torch
    n = la_ce_workspace_bytes(N, V, d, ce_chunk)
    if n == 0:
        raise ValueError(f"invalid shape N={N} V={V} d={d} ce_chunk={ce_chunk}")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _ce_args(h, W, targets):
    import torch
    if h.dim() != 2 or W.dim() != 2 or h.shape[1] != W.shape[1]:
        raise ValueError(f"h [N, d] and W [V, d] expected, got {tuple(h.shape)} and {tuple(W.shape)}")
    N, d = h.shape
    _check_tensor("h", h, h.shape, torch.bfloat16, h.device)
    _check_tensor("W", W, W.shape, torch.bfloat16, h.device)
    _check_tensor("targets", targets, torch.Size((N,)), torch.int32, h.device)
    return N, W.shape[0], d


def ce_fwd(h, W, targets, *, ce_chunk: int = 512, workspace=None, stream=None):
    """Chunked cross-entropy of the tied head: returns (loss (0-d float32 tensor), lse [N])."""
    import torch
    N, V, d = _ce_args(h, W, targets)
    if workspace is None:
        workspace = ce_workspace(N, V, d, ce_chunk, h.device)
    loss = torch.empty((), dtype=torch.float32, device=h.device)
    lse = torch.empty(N, dtype=torch.float32, device=h.device)
    la_ce_fwd(h, W, targets, N, V, d, ce_chunk, loss, lse, workspace, workspace.numel(), _stream(stream))
    return loss, lse


def ce_bwd(h, W, targets, lse, dloss: float = 1.0, *, ce_chunk: int = 512, workspace=None, stream=None):
    """Gradients of dloss * ce_fwd's loss: returns (dh bf16 [N, d], dW float32 [V, d])."""
    import torch
    N, V, d = _ce_args(h, W, targets)
    _check_tensor("lse", lse, torch.Size((N,)), torch.float32, h.device)
    if workspace is None:
        workspace = ce_workspace(N, V, d, ce_chunk, h.device)
    dh = torch.empty_like(h)
    dW = torch.empty(V, d, dtype=torch.float32, device=h.device)
    la_ce_bwd(h, W, targets, lse, float(dloss), N, V, d, ce_chunk, dh, dW, workspace, workspace.numel(),
              _stream(stream))
    return dh, dW


def cumsum_fwd(q, k, v, S0=None, z0=None, *, eps: float = 1e-6, o=None, S_out=None, z_out=None, stream=None):
    """The cumsum form of chunked_fwd (token-by-token scan, fp32 state on chip, CUDA
    cores).  Returns (o, S_out, z_out)."""
    import torch
    G, C, D = q.shape
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(n, t, q.shape, q.dtype, q.device)
    for n, t, shp in (("S0", S0, (G, D, D)), ("z0", z0, (G, D))):
        if t is not None:
            _check_tensor(n, t, torch.Size(shp), torch.float32, q.device)
    o = torch.empty_like(q) if o is None else o
    S_out = torch.empty(G, D, D, device=q.device, dtype=torch.float32) if S_out is None else S_out
    z_out = torch.empty(G, D, device=q.device, dtype=torch.float32) if z_out is None else z_out
    la_cumsum_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, _dtype_code(q), eps, _stream(stream))
    return o, S_out, z_out


def cumsum_bwd(q, k, v, S0, z0, dO, dS_out=None, dz_out=None, *, eps: float = 1e-6, out: Optional[tuple] = None,
               workspace=None, stream=None):
    """The cumsum form of chunked_bwd.  `workspace` (a CUDA tensor of at least
    la_cumsum_bwd_workspace_bytes bytes) is allocated here when not given.  Returns
    (dq, dk, dv, dS0, dz0)."""
    import torch
    G, C, D = q.shape
    dq, dk, dv, dS0, dz0 = _bwd_args(q, k, v, S0, z0, dO, dS_out, dz_out, out)
    need = la_cumsum_bwd_workspace_bytes(G, C, D, _dtype_code(q))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    la_cumsum_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, D, _dtype_code(q), eps, workspace,
                  wbytes, _stream(stream))
    return dq, dk, dv, dS0, dz0


def chunked_bwd_split(q, k, v, S0, z0, dO, dS_out=None, dz_out=None, *, block: int = 64, eps: float = 1e-6,
                      out: Optional[tuple] = None, workspace=None, stream=None):
    """chunked_bwd cut along the tokens for few groups of long chunks (bf16, D = 64 or 128): the
    pieces of every group run on separate CTAs, between prefix sums over the pieces in
    token order (the forward carries) and in reverse (the carry gradients).  `workspace`
    (a CUDA tensor of at least la_bwd_split_workspace_bytes bytes) is allocated here when
    not given.  Returns (dq, dk, dv, dS0, dz0)."""
    import torch
    G, C, D = q.shape
    dq, dk, dv, dS0, dz0 = _bwd_args(q, k, v, S0, z0, dO, dS_out, dz_out, out)
    need = la_bwd_split_workspace_bytes(G, C, D, _dtype_code(q))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    la_chunked_bwd_split(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, D, block, _dtype_code(q),
                         eps, workspace, wbytes, _stream(stream))
    return dq, dk, dv, dS0, dz0


def chunked_bwd(q, k, v, S0, z0, dO, dS_out=None, dz_out=None, *, block: int = 64, eps: float = 1e-6,
                out: Optional[tuple] = None, stream=None):
    """Backward of chunked_fwd, recomputed from its inputs.  Returns (dq, dk, dv, dS0, dz0)."""
    import torch
    G, C, D = q.shape
    dt = q.dtype
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _check_tensor(n, t, q.shape, dt, q.device)
    for n, t, shp in (("S0", S0, (G, D, D)), ("z0", z0, (G, D)), ("dS_out", dS_out, (G, D, D)),
                      ("dz_out", dz_out, (G, D))):
        if t is not None:
            _check_tensor(n, t, torch.Size(shp), torch.float32, q.device)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q),
               torch.empty(G, D, D, device=q.device, dtype=torch.float32),
               torch.empty(G, D, device=q.device, dtype=torch.float32))
    dq, dk, dv, dS0, dz0 = out
    la_chunked_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, D, block,
                   _dtype_code(q), eps, _stream(stream))
    return dq, dk, dv, dS0, dz0


def step_workspace(G: int, C: int, D: int, dtype, device=None):
    """Device workspace (uint8 CUDA tensor) for chunked_step_host on this shape."""
    import torch
    code = LA_BF16 if dtype == torch.bfloat16 else LA_F32 if dtype == torch.float32 else None
    if code is None:
        raise TypeError(f"dtype must be bfloat16 or float32, got {dtype}")
    n = la_step_workspace_bytes(G, C, D, code)
    if n == 0 and G * C * D > 0:
        raise ValueError(f"unsupported shape G={G} C={C} D={D}")
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")


def chunked_step_host(q, k, v, S0, z0, dO, dS_out=None, dz_out=None, *, out, workspace, block: int = 64,
                      eps: float = 1e-6, stream=None):
    """Forward + backward of one chunk with HOST tensors (CPU, ideally pinned): copies the
    inputs into `workspace` (from step_workspace), runs the two kernels and copies the
    results into `out` = (o, S_out, z_out, dq, dk, dv, dS0, dz0) (CPU tensors; the carry
    entries may be None), all on `stream`.  The results are valid once the stream is done."""
    import torch
    G, C, D = q.shape
    dt = q.dtype
    cpu = torch.device("cpu")
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _check_tensor(n, t, q.shape, dt, cpu)
    for n, t, shp in (("S0", S0, (G, D, D)), ("z0", z0, (G, D)), ("dS_out", dS_out, (G, D, D)),
                      ("dz_out", dz_out, (G, D))):
        if t is not None:
            _check_tensor(n, t, torch.Size(shp), torch.float32, cpu)
    o, S_out, z_out, dq, dk, dv, dS0, dz0 = out
    for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_tensor(n, t, q.shape, dt, cpu)
    for n, t, shp in (("S_out", S_out, (G, D, D)), ("z_out", z_out, (G, D)), ("dS0", dS0, (G, D, D)),
                      ("dz0", dz0, (G, D))):
        if t is not None:
            _check_tensor(n, t, torch.Size(shp), torch.float32, cpu)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    la_chunked_step_host(q, k, v, S0, z0, dO, dS_out, dz_out, o, S_out, z_out, dq, dk, dv, dS0, dz0,
                         workspace, workspace.numel() * workspace.element_size(), G, C, D, block,
                         _dtype_code(q), eps, _stream(stream) if stream is not None else
                         torch.cuda.current_stream(workspace.device).cuda_stream)
    return out
