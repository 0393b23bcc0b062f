"""The chunk-parallel forward without a workspace (la_chunked_fwd_split_static).

It runs the same kernels as la_chunked_fwd_split on a module-level device array, so on
the same inputs its results must equal the workspace form bit for bit, call after call.
(The file name puts it after the other GPU tests; it also passes on its own.)"""
import pytest
import torch

import causal_linear_attention_gb300 as la
from causal_linear_attention_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
EPS = 1e-6


def test_static_scratch_forward_equals_the_workspace_form_on_consecutive_calls():
    """Two calls in a row with different plans, issued back to back on one stream before a
    single synchronisation: the second reuses the module array the first has just used, and
    each must still equal its workspace-form result bit for bit."""
    la.build()
    cases = ((2, 4096, 31), (8, 1000, 32))
    refs, outs = [], []
    for G, C, seed in cases:
        assert la.la_fwd_split_workspace_bytes(G, C, 64, la.LA_BF16) > 0
        x = make_inputs(G, C, 64, dtype="bf16", seed=seed, carry=True).to(DEV)
        refs.append(la.chunked_fwd_split(x.q, x.k, x.v, x.S0, x.z0, block=64, eps=EPS))
        outs.append((x, torch.empty_like(x.q), torch.empty(G, 64, 64, device=DEV), torch.empty(G, 64, device=DEV)))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for (G, C, _), (x, o, S, z) in zip(cases, outs):
        la.la_chunked_fwd_split_static(x.q, x.k, x.v, x.S0, x.z0, o, S, z, G, C, 64, 64, la.LA_BF16, EPS, stream)
    torch.cuda.synchronize()
    for ref, (x, o, S, z) in zip(refs, outs):
        for name, a, b in zip(("o", "S_out", "z_out"), (o, S, z), ref):
            assert torch.equal(a, b), name
    assert la.la_device_status() == 0


def test_static_scratch_forward_without_a_split_is_the_plain_forward():
    x = make_inputs(200, 256, 64, dtype="bf16", seed=33, carry=True).to(DEV)
    assert la.la_fwd_split_workspace_bytes(200, 256, 64, la.LA_BF16) == 0
    ref = la.chunked_fwd(x.q, x.k, x.v, x.S0, x.z0, block=64, eps=EPS)
    o = torch.empty_like(x.q)
    S = torch.empty(200, 64, 64, device=DEV)
    z = torch.empty(200, 64, device=DEV)
    la.la_chunked_fwd_split_static(x.q, x.k, x.v, x.S0, x.z0, o, S, z, 200, 256, 64, 64, la.LA_BF16, EPS,
                                   torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    for a, b in zip((o, S, z), ref):
        assert torch.equal(a, b)


def test_static_scratch_forward_at_head_size_128():
    """Head size 128: where the module array holds the workspace form's plan (64 cells of
    66,048 bytes) the results are the same bits; where it does not (G = 1, C = 16384 asks
    for 128 pieces, the array holds 127) the plan is cut to fit and the results match the
    oracle within the bf16 bounds."""
    import oracle
    import numpy as np
    x = make_inputs(2, 4096, 128, dtype="bf16", seed=35, carry=True).to(DEV)
    ref = la.chunked_fwd_split(x.q, x.k, x.v, x.S0, x.z0, block=64, eps=EPS)
    o = torch.empty_like(x.q)
    S = torch.empty(2, 128, 128, device=DEV)
    z = torch.empty(2, 128, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    la.la_chunked_fwd_split_static(x.q, x.k, x.v, x.S0, x.z0, o, S, z, 2, 4096, 128, 64, la.LA_BF16, EPS, stream)
    torch.cuda.synchronize()
    for name, a, b in zip(("o", "S_out", "z_out"), (o, S, z), ref):
        assert torch.equal(a, b), name
    h = make_inputs(1, 16384, 128, dtype="bf16", seed=36, carry=True)
    x = h.to(DEV)
    o = torch.empty_like(x.q)
    S = torch.empty(1, 128, 128, device=DEV)
    z = torch.empty(1, 128, device=DEV)
    la.la_chunked_fwd_split_static(x.q, x.k, x.v, x.S0, x.z0, o, S, z, 1, 16384, 128, 64, la.LA_BF16, EPS, stream)
    torch.cuda.synchronize()
    ro, rS, rz = oracle.fwd(h.q, h.k, h.v, h.S0, h.z0, eps=EPS)
    for name, a, r, tol in (("o", o, ro, 2e-2), ("S_out", S, rS, 1e-2), ("z_out", z, rz, 1e-2)):
        a = a.double().cpu().numpy()
        assert np.abs(a - r).max() / np.abs(r).max() < tol, name
    assert la.la_device_status() == 0
