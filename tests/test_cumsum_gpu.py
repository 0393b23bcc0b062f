"""GPU parity of the cumsum form (la_cumsum_fwd / la_cumsum_bwd, a token-by-token scan)
against the fp64 oracle, through the C ABI.  Shapes: the Fractus-1B block (G = 160,
C = 128, D = 64), wide heads (D = 128), ragged chunks (C not a multiple of the 32-token
staging block), the empty and one-token chunks; inputs from the shared seeded
generator.  Metric and tolerances: tests/parity_util.py."""
import pytest
import torch

import causal_linear_attention_gb300 as la
import oracle
from causal_linear_attention_gb300.inputs import make_inputs
from parity_util import check, max_rel

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
EPS = 1e-6
FWD_NAMES = ("o", "S_out", "z_out")
BWD_NAMES = ("dq", "dk", "dv", "dS0", "dz0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    la.build()
    oracle.build()
    yield


def fwd_bwd(G, C, D, dtype, seed, carry=True, upstream=True):
    x = make_inputs(G, C, D, dtype=dtype, seed=seed, carry=carry, grads=True)
    if not upstream:
        x.dS_out = x.dz_out = None
    d = x.to(DEV)
    got_f = la.cumsum_fwd(d.q, d.k, d.v, d.S0, d.z0, eps=EPS)
    got_b = la.cumsum_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, eps=EPS)
    torch.cuda.synchronize()
    assert la.la_device_status() == 0
    check(got_f, oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS), dtype, FWD_NAMES)
    check(got_b, oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS), dtype, BWD_NAMES)
    return x, d, got_f, got_b


@pytest.mark.parametrize("G,C,D,dtype", [
    (8, 128, 64, "f32"),      # the fp32 workload: 1e-4
    (160, 128, 64, "bf16"),   # the Fractus-1B block
    (4, 200, 128, "bf16"),    # wide heads, ragged
    (3, 200, 128, "f32"),
    (5, 33, 64, "bf16"),      # one token past a staging block
    (2, 1, 64, "f32"),        # one token
    (2, 1000, 64, "bf16"),    # several staging blocks, ragged
    (160, 128, 128, "bf16"),  # wide heads over many groups: two forward CTAs per group, three per SM
])
def test_cumsum_matches_oracle(G, C, D, dtype):
    fwd_bwd(G, C, D, dtype, seed=G * 1000 + C)


def test_cumsum_without_carry_or_upstream_gradient():
    fwd_bwd(3, 100, 64, "bf16", seed=7, carry=False, upstream=False)


def test_cumsum_empty_chunk_passes_the_carry_through():
    x = make_inputs(3, 0, 64, dtype="f32", seed=8, carry=True, grads=True)
    d = x.to(DEV)
    o, S, z = la.cumsum_fwd(d.q, d.k, d.v, d.S0, d.z0, eps=EPS)
    dq, dk, dv, dS0, dz0 = la.cumsum_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, eps=EPS)
    torch.cuda.synchronize()
    assert o.numel() == 0 and dq.numel() == 0
    assert torch.equal(S.cpu(), x.S0) and torch.equal(z.cpu(), x.z0)
    assert torch.equal(dS0.cpu(), x.dS_out) and torch.equal(dz0.cpu(), x.dz_out)


@pytest.mark.parametrize("G,C,D,dtype", [(4, 150, 64, "bf16"), (3, 33, 128, "f32")])
def test_cumsum_in_place_carries(G, C, D, dtype):
    """S_out over S0, z_out over z0 (forward); dS0 over dS_out, dz0 over dz_out (backward:
    the dv sweep then reads the workspace's copy of dS_out, which starts on a 16-byte
    boundary after the 2 G C per-token values, 198 floats in the second case)."""
    x = make_inputs(G, C, D, dtype=dtype, seed=9, carry=True, grads=True)
    d = x.to(DEV)
    S, z = d.S0.clone(), d.z0.clone()
    got = la.cumsum_fwd(d.q, d.k, d.v, S, z, eps=EPS, S_out=S, z_out=z)
    dS, dz = d.dS_out.clone(), d.dz_out.clone()
    out = (torch.empty_like(d.q), torch.empty_like(d.q), torch.empty_like(d.q), dS, dz)
    gotb = la.cumsum_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, dS, dz, eps=EPS, out=out)
    torch.cuda.synchronize()
    check(got, oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS), dtype, FWD_NAMES)
    check(gotb, oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS), dtype, BWD_NAMES)


def test_cumsum_agrees_with_the_chunked_kernels():
    """The two implementations of the same definition, side by side (bf16 bounds)."""
    x, d, got_f, got_b = fwd_bwd(16, 256, 64, "bf16", seed=11)
    ch_f = la.chunked_fwd(d.q, d.k, d.v, d.S0, d.z0, block=64, eps=EPS)
    ch_b = la.chunked_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=64, eps=EPS)
    torch.cuda.synchronize()
    for a, b, n in zip(got_f + got_b, ch_f + ch_b, FWD_NAMES + BWD_NAMES):
        assert max_rel(a, b) < 2e-2, n


def test_cumsum_is_deterministic():
    x = make_inputs(6, 300, 128, dtype="bf16", seed=12, carry=True, grads=True)
    d = x.to(DEV)
    a = la.cumsum_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, eps=EPS)
    b = la.cumsum_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, eps=EPS)
    torch.cuda.synchronize()
    for u, w in zip(a, b):
        assert torch.equal(u, w)
