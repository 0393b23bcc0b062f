"""Pins of oracle/torch_chunked.py (the PyTorch-CPU restatement of the page's chunked form,
the bench's like-for-like CPU baseline): run in float64 it equals the fp64 per-token oracle
(itself pinned in test_oracle_pins.py) forward and backward at every block size, including
ragged last blocks; in float32 it stays within fp32 rounding of it."""
import numpy as np
import pytest
import torch

import oracle
from oracle import torch_chunked
from causal_linear_attention_gb300.inputs import make_inputs


def _t(a, dtype):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dtype)


def _rel(a, b):
    a = a.detach().double().numpy() if isinstance(a, torch.Tensor) else a
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("G,C,D,block", [(2, 100, 16, 32), (3, 64, 8, 64), (1, 37, 8, 5), (2, 130, 16, 128)])
def test_float64_equals_the_token_oracle(G, C, D, block):
    x = make_inputs(G, C, D, dtype="fp32", seed=G * C + block, carry=True, grads=True)
    args = [_t(getattr(x, n), torch.float64) for n in ("q", "k", "v", "S0", "z0", "dO", "dS_out", "dz_out")]
    got = torch_chunked.chunked_fwd_bwd(*args, block=block, eps=1e-6)
    ref = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=1e-6) + \
        oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=1e-6)
    for n, a, b in zip(("o", "S_out", "z_out", "dq", "dk", "dv", "dS0", "dz0"), got, ref):
        assert _rel(a, b) < 1e-10, n


def test_float32_within_rounding_and_no_carry():
    x = make_inputs(2, 256, 64, dtype="fp32", seed=7, carry=False, grads=True)
    q, k, v, dO = (_t(getattr(x, n), torch.float32) for n in ("q", "k", "v", "dO"))
    o, S, z = torch_chunked.chunked_fwd(q, k, v, None, None, block=64, eps=1e-6)
    ro, rS, rz = oracle.fwd(x.q, x.k, x.v, None, None, eps=1e-6)
    assert _rel(o, ro) < 1e-4 and _rel(S, rS) < 1e-5 and _rel(z, rz) < 1e-5
