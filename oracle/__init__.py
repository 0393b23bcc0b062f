"""fp64 CPU oracle for causal linear attention with a carried running state.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It shares
no code with the CUDA path (``causal_linear_attention_gb300``) and imports nothing
from it; the two meet only in the seeded input generator, which holds none of the
method's arithmetic.

Method source: "Fractus-1B training optimization -- 2026-08-22" (section 1,
"Bottleneck #1": the state is a causal cumsum of outer products, written on the
page as the masked einsum ``"tj,bjpq->btpq"``; the derivative of a cumsum is a
reverse cumsum.  Section 2, "Opt 2": the chunked form with a masked block x block
score matrix inside a block and the running state (S_run, z_run) across blocks,
updated inclusively AFTER reading.  Section 2, "Opt 6": the carry (S, z) is
threaded from chunk to chunk).

The page prints no output normalisation.  Reading used throughout:

    S_t = S0 + sum_{j<=t} k_j v_j^T        (S[p][c]: p = key dim, c = value dim)
    z_t = z0 + sum_{j<=t} k_j
    o_t = (q_t^T S_t) / (q_t . z_t + eps)

Functions (numpy float64, row-major; q, k, v, o, dO: [G, C, D]; S: [G, D, D];
z: [G, D]; ``None`` carries / upstream carry grads mean zeros):

* ``fwd``            per-token loop (C, OpenMP over groups) -- the definition.
* ``bwd``            per-token reverse-cumsum backward of ``fwd`` (C).
* ``fwd_chunked``    the page's chunked form with a block size (C).
* ``bwd_chunked``    the chunked backward (forward sweep + reverse sweep) (C).
* ``fwd_einsum``     the page's masked-einsum form, O(C^2 D^2) memory; tiny inputs.
* ``torch_chunked``  (submodule) the chunked form as PyTorch CPU ops, fp32 or fp64, the backward
                   by autograd: the bench's like-for-like CPU number (the page times its own
                   chunked form this way).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(hand-derived golden values, closed forms, invariants, finite differences and
float64 autograd of the einsum form).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblaoracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile la_oracle.c into a shared library (gcc, OpenMP, fp64)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        Dbl = ctypes.c_double
        lib.la_oracle_threads.restype = I
        lib.la_oracle_fwd.argtypes = [I, I, I, P, P, P, P, P, Dbl, P, P, P]
        lib.la_oracle_fwd.restype = None
        lib.la_oracle_fwd_chunked.argtypes = [I, I, I, I, P, P, P, P, P, Dbl, P, P, P]
        lib.la_oracle_fwd_chunked.restype = None
        lib.la_oracle_bwd.argtypes = [I, I, I, P, P, P, P, P, P, P, P, Dbl, P, P, P, P, P]
        lib.la_oracle_bwd.restype = None
        lib.la_oracle_bwd_chunked.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, Dbl,
                                              P, P, P, P, P]
        lib.la_oracle_bwd_chunked.restype = None
        _lib = lib
        return lib


def threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().la_oracle_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _shapes(q, k, v):
    if q.ndim != 3 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError(f"q, k, v must share one [G, C, D] shape, got {q.shape}, {k.shape}, {v.shape}")
    return q.shape


def _check_carry(S, z, G, D):
    if S is not None and S.shape != (G, D, D):
        raise ValueError(f"S must be [G, D, D] = {(G, D, D)}, got {S.shape}")
    if z is not None and z.shape != (G, D):
        raise ValueError(f"z must be [G, D] = {(G, D)}, got {z.shape}")


def fwd(q, k, v, S0=None, z0=None, eps=1e-6):
    """Per-token forward (the definition).  Returns (o, S_out, z_out)."""
    q, k, v, S0, z0 = (_f64(x) for x in (q, k, v, S0, z0))
    G, C, D = _shapes(q, k, v)
    _check_carry(S0, z0, G, D)
    o = np.empty((G, C, D))
    S_out = np.empty((G, D, D))
    z_out = np.empty((G, D))
    _load().la_oracle_fwd(G, C, D, _ptr(q), _ptr(k), _ptr(v), _ptr(S0), _ptr(z0),
                          float(eps), _ptr(o), _ptr(S_out), _ptr(z_out))
    return o, S_out, z_out


def fwd_chunked(q, k, v, S0=None, z0=None, eps=1e-6, block=64):
    """The page's chunked forward with the given block size.  Returns (o, S_out, z_out)."""
    q, k, v, S0, z0 = (_f64(x) for x in (q, k, v, S0, z0))
    G, C, D = _shapes(q, k, v)
    _check_carry(S0, z0, G, D)
    if block < 1:
        raise ValueError("block must be >= 1")
    o = np.empty((G, C, D))
    S_out = np.empty((G, D, D))
    z_out = np.empty((G, D))
    _load().la_oracle_fwd_chunked(G, C, D, int(block), _ptr(q), _ptr(k), _ptr(v), _ptr(S0),
                                  _ptr(z0), float(eps), _ptr(o), _ptr(S_out), _ptr(z_out))
    return o, S_out, z_out


def bwd(q, k, v, S0, z0, dO, dS_out=None, dz_out=None, eps=1e-6):
    """Per-token backward.  Returns (dq, dk, dv, dS0, dz0)."""
    q, k, v, S0, z0, dO, dS_out, dz_out = (_f64(x) for x in (q, k, v, S0, z0, dO, dS_out, dz_out))
    G, C, D = _shapes(q, k, v)
    _check_carry(S0, z0, G, D)
    _check_carry(dS_out, dz_out, G, D)
    if dO.shape != q.shape:
        raise ValueError("dO must match q")
    dq, dk, dv = (np.empty((G, C, D)) for _ in range(3))
    dS0 = np.empty((G, D, D))
    dz0 = np.empty((G, D))
    _load().la_oracle_bwd(G, C, D, _ptr(q), _ptr(k), _ptr(v), _ptr(S0), _ptr(z0), _ptr(dO),
                          _ptr(dS_out), _ptr(dz_out), float(eps), _ptr(dq), _ptr(dk), _ptr(dv),
                          _ptr(dS0), _ptr(dz0))
    return dq, dk, dv, dS0, dz0


def bwd_chunked(q, k, v, S0, z0, dO, dS_out=None, dz_out=None, eps=1e-6, block=64):
    """Chunked backward (forward sweep, then reverse sweep).  Returns (dq, dk, dv, dS0, dz0)."""
    q, k, v, S0, z0, dO, dS_out, dz_out = (_f64(x) for x in (q, k, v, S0, z0, dO, dS_out, dz_out))
    G, C, D = _shapes(q, k, v)
    _check_carry(S0, z0, G, D)
    _check_carry(dS_out, dz_out, G, D)
    dq, dk, dv = (np.empty((G, C, D)) for _ in range(3))
    dS0 = np.empty((G, D, D))
    dz0 = np.empty((G, D))
    _load().la_oracle_bwd_chunked(G, C, D, int(block), _ptr(q), _ptr(k), _ptr(v), _ptr(S0),
                                  _ptr(z0), _ptr(dO), _ptr(dS_out), _ptr(dz_out), float(eps),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dS0), _ptr(dz0))
    return dq, dk, dv, dS0, dz0


def fwd_einsum(q, k, v, S0=None, z0=None, eps=1e-6):
    """The page's masked-einsum form (section 1, "Bottleneck #1"): materialise every
    outer product k_j v_j^T, then S_t = S0 + einsum("tj,gjpq->gtpq", tril, outer).
    O(C^2 D^2) work and O(C D^2) memory per group: tiny inputs only."""
    q, k, v, S0, z0 = (_f64(x) for x in (q, k, v, S0, z0))
    G, C, D = _shapes(q, k, v)
    if G * C * C * D * D > 5e7:
        raise ValueError("fwd_einsum is for tiny inputs only")
    if C == 0:
        S_fin = np.zeros((G, D, D)) if S0 is None else S0.copy()
        z_fin = np.zeros((G, D)) if z0 is None else z0.copy()
        return np.zeros((G, 0, D)), S_fin, z_fin
    outer = np.einsum("gjp,gjq->gjpq", k, v)
    mask = np.tril(np.ones((C, C)))
    S = np.einsum("tj,gjpq->gtpq", mask, outer)
    z = np.einsum("tj,gjp->gtp", mask, k)
    if S0 is not None:
        S = S + S0[:, None]
    if z0 is not None:
        z = z + z0[:, None]
    num = np.einsum("gtp,gtpq->gtq", q, S)
    den = np.einsum("gtp,gtp->gt", q, z) + eps
    return num / den[..., None], S[:, -1], z[:, -1]
