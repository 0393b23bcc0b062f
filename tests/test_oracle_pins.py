"""Pins for the fp64 oracle, checked against things other than the oracle itself.

Source of the method: "Fractus-1B training optimization -- 2026-08-22", section 1
("Bottleneck #1": masked-einsum form, cumsum form, reverse-cumsum derivative) and
section 2 ("Opt 1" looped-reference / einsum equivalence proofs, "Opt 2" chunked
form, "Opt 6" carry evolution across consecutive chunks).

Each pin is chosen so that a plausible slip in the oracle (exclusive instead of
inclusive state, transposed outer product, a dropped carry or eps term, a wrong
sign in the reverse cumsum) fails at least one of them:

* hand-worked golden values (tests/golden/hand_examples.json)
* per-token loop == masked einsum == chunked form for several block sizes
* closed forms for the final carry, S_out = S0 + K^T V and z_out = z0 + K^T 1
* carry threading: two chunks with the carry passed on == one chunk of 2C
* linearity in (v, S0), homogeneity at eps = 0, a causal running-mean special case
* backward: central finite differences, float64 autograd of the einsum form,
  chunked backward == per-token backward, gradient carry threading
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from causal_linear_attention_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _rand(G, C, D, seed, carry=True, grads=False):
    inp = make_inputs(G, C, D, dtype="f32", seed=seed, carry=carry, grads=grads)
    return {k: v.double().numpy() for k, v in inp.tensors().items()}


def _arr(x, shape=None):
    return None if x is None else np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------- golden values

@pytest.mark.parametrize("name", ["scalar_carry_eps1", "orientation_d2"])
def test_golden_forward(name):
    ex = json.load(open(GOLDEN))[name]
    q, k, v = (_arr(ex[n])[None] for n in ("q", "k", "v"))
    S0 = None if ex["S0"] is None else _arr(ex["S0"])[None]
    z0 = None if ex["z0"] is None else _arr(ex["z0"])[None]
    for f in (oracle.fwd, lambda *a, **kw: oracle.fwd_chunked(*a, block=1, **kw),
              lambda *a, **kw: oracle.fwd_chunked(*a, block=64, **kw), oracle.fwd_einsum):
        o, S, z = f(q, k, v, S0, z0, eps=ex["eps"])
        np.testing.assert_allclose(o[0], ex["o"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(S[0], ex["S_out"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(z[0], ex["z_out"], rtol=0, atol=1e-14)


def test_golden_backward():
    ex = json.load(open(GOLDEN))["scalar_carry_eps1"]
    a = {n: _arr(ex[n])[None] for n in ("q", "k", "v", "S0", "z0", "dO", "dS_out", "dz_out")}
    for f in (oracle.bwd, lambda *x, **kw: oracle.bwd_chunked(*x, block=1, **kw),
              lambda *x, **kw: oracle.bwd_chunked(*x, block=2, **kw)):
        dq, dk, dv, dS0, dz0 = f(a["q"], a["k"], a["v"], a["S0"], a["z0"], a["dO"],
                                 a["dS_out"], a["dz_out"], eps=ex["eps"])
        for got, name in ((dq, "dq"), (dk, "dk"), (dv, "dv"), (dS0, "dS0"), (dz0, "dz0")):
            np.testing.assert_allclose(got[0], ex[name], rtol=0, atol=1e-14, err_msg=name)


# ---------------------------------------------------------------- forward forms agree

@pytest.mark.parametrize("G,C,D", [(2, 9, 3), (3, 16, 4), (1, 13, 5)])
def test_loop_equals_einsum_and_chunked(G, C, D):
    x = _rand(G, C, D, seed=G * 100 + C)
    ref = oracle.fwd_einsum(x["q"], x["k"], x["v"], x["S0"], x["z0"], eps=1e-6)
    outs = [oracle.fwd(x["q"], x["k"], x["v"], x["S0"], x["z0"], eps=1e-6)]
    for block in (1, 2, 4, 7, 64, C):
        outs.append(oracle.fwd_chunked(x["q"], x["k"], x["v"], x["S0"], x["z0"], eps=1e-6, block=block))
    for o, S, z in outs:
        np.testing.assert_allclose(o, ref[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(S, ref[1], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(z, ref[2], rtol=1e-12, atol=1e-12)


def test_no_carry_equals_zero_carry():
    x = _rand(2, 11, 4, seed=5)
    a = oracle.fwd(x["q"], x["k"], x["v"], None, None)
    b = oracle.fwd(x["q"], x["k"], x["v"], np.zeros((2, 4, 4)), np.zeros((2, 4)))
    for u, w in zip(a, b):
        np.testing.assert_array_equal(u, w)


def test_empty_chunk_passes_carry_through():
    x = _rand(2, 3, 4, seed=6)
    q = np.zeros((2, 0, 4))
    o, S, z = oracle.fwd(q, q, q, x["S0"], x["z0"])
    assert o.shape == (2, 0, 4)
    np.testing.assert_array_equal(S, x["S0"])
    np.testing.assert_array_equal(z, x["z0"])


# ---------------------------------------------------------------- closed forms / invariants

def test_final_carry_closed_form():
    x = _rand(3, 37, 8, seed=7)
    _, S, z = oracle.fwd(x["q"], x["k"], x["v"], x["S0"], x["z0"])
    S_ref = x["S0"] + np.matmul(x["k"].transpose(0, 2, 1), x["v"])
    z_ref = x["z0"] + x["k"].sum(axis=1)
    np.testing.assert_allclose(S, S_ref, rtol=1e-12, atol=1e-11)
    np.testing.assert_allclose(z, z_ref, rtol=1e-12, atol=1e-11)


@pytest.mark.parametrize("split", [1, 17, 40])
def test_carry_threading_equals_one_pass(split):
    x = _rand(2, 41, 6, seed=8)
    full = oracle.fwd(x["q"], x["k"], x["v"], x["S0"], x["z0"])
    a = oracle.fwd(x["q"][:, :split], x["k"][:, :split], x["v"][:, :split], x["S0"], x["z0"])
    b = oracle.fwd(x["q"][:, split:], x["k"][:, split:], x["v"][:, split:], a[1], a[2])
    np.testing.assert_allclose(np.concatenate([a[0], b[0]], axis=1), full[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b[1], full[1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b[2], full[2], rtol=1e-12, atol=1e-12)


def test_linearity_in_v_and_S0():
    x = _rand(2, 15, 5, seed=9)
    y = _rand(2, 15, 5, seed=10)
    al, be = 0.7, -1.3
    f = lambda v, S0: oracle.fwd(x["q"], x["k"], v, S0, x["z0"], eps=1e-3)
    o1, S1, z1 = f(x["v"], x["S0"])
    o2, S2, z2 = f(y["v"], y["S0"])
    o3, S3, z3 = f(al * x["v"] + be * y["v"], al * x["S0"] + be * y["S0"])
    np.testing.assert_allclose(o3, al * o1 + be * o2, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(S3, al * S1 + be * S2, rtol=1e-11, atol=1e-10)
    np.testing.assert_array_equal(z1, z3)  # z does not depend on v


def test_homogeneity_at_zero_eps():
    x = _rand(2, 12, 4, seed=11)
    o, _, _ = oracle.fwd(x["q"], x["k"], x["v"], x["S0"], x["z0"], eps=0.0)
    o_q, _, _ = oracle.fwd(3.5 * x["q"], x["k"], x["v"], x["S0"], x["z0"], eps=0.0)
    o_k, _, _ = oracle.fwd(x["q"], 0.25 * x["k"], x["v"], 0.25 * x["S0"], 0.25 * x["z0"], eps=0.0)
    np.testing.assert_allclose(o_q, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o_k, o, rtol=1e-12, atol=1e-12)


def test_running_mean_special_case():
    """q = k = 1, no carry: o_t = D * sum_{j<=t} v_j / (D (t+1) + eps), a causal mean."""
    G, C, D, eps = 2, 19, 6, 1e-3
    v = _rand(G, C, D, seed=12)["v"]
    ones = np.ones((G, C, D))
    o, _, _ = oracle.fwd(ones, ones, v, None, None, eps=eps)
    t = np.arange(1, C + 1)[None, :, None]
    ref = D * np.cumsum(v, axis=1) / (D * t + eps)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward

def _loss(q, k, v, S0, z0, dO, dS, dz, eps):
    o, S, z = oracle.fwd(q, k, v, S0, z0, eps=eps)
    return float((o * dO).sum() + (S * dS).sum() + (z * dz).sum())


def test_backward_finite_differences():
    G, C, D, eps = 2, 7, 3, 1e-2
    x = _rand(G, C, D, seed=13, grads=True)
    args = [x["q"], x["k"], x["v"], x["S0"], x["z0"]]
    grads = oracle.bwd(*args, x["dO"], x["dS_out"], x["dz_out"], eps=eps)
    h = 1e-6
    for ai, (arr, g) in enumerate(zip(args, grads)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            keep = arr[idx]
            arr[idx] = keep + h
            lp = _loss(*args, x["dO"], x["dS_out"], x["dz_out"], eps)
            arr[idx] = keep - h
            lm = _loss(*args, x["dO"], x["dS_out"], x["dz_out"], eps)
            arr[idx] = keep
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7, err_msg=f"argument {ai}")


def _torch_einsum_forward(q, k, v, S0, z0, eps):
    """Independent float64 formulation for autograd: the page's masked einsum."""
    C = q.shape[1]
    outer = torch.einsum("gjp,gjq->gjpq", k, v)
    mask = torch.tril(torch.ones(C, C, dtype=torch.float64))
    S = torch.einsum("tj,gjpq->gtpq", mask, outer) + S0[:, None]
    z = torch.einsum("tj,gjp->gtp", mask, k) + z0[:, None]
    o = torch.einsum("gtp,gtpq->gtq", q, S) / (torch.einsum("gtp,gtp->gt", q, z) + eps)[..., None]
    return o, S[:, -1], z[:, -1]


@pytest.mark.parametrize("G,C,D", [(2, 9, 4), (1, 20, 3)])
def test_backward_matches_float64_autograd(G, C, D):
    eps = 1e-6
    x = _rand(G, C, D, seed=14 + C, grads=True)
    t = {n: torch.tensor(x[n], requires_grad=n in ("q", "k", "v", "S0", "z0")) for n in x}
    o, S, z = _torch_einsum_forward(t["q"], t["k"], t["v"], t["S0"], t["z0"], eps)
    loss = (o * t["dO"]).sum() + (S * t["dS_out"]).sum() + (z * t["dz_out"]).sum()
    loss.backward()
    ref = [t[n].grad.numpy() for n in ("q", "k", "v", "S0", "z0")]
    for got in (oracle.bwd(x["q"], x["k"], x["v"], x["S0"], x["z0"], x["dO"], x["dS_out"], x["dz_out"], eps=eps),
                oracle.bwd_chunked(x["q"], x["k"], x["v"], x["S0"], x["z0"], x["dO"], x["dS_out"],
                                   x["dz_out"], eps=eps, block=4)):
        for g, r, name in zip(got, ref, ("dq", "dk", "dv", "dS0", "dz0")):
            np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-10, err_msg=name)


@pytest.mark.parametrize("block", [1, 3, 8, 64])
def test_chunked_backward_equals_token_backward(block):
    x = _rand(3, 23, 5, seed=15, grads=True)
    a = oracle.bwd(x["q"], x["k"], x["v"], x["S0"], x["z0"], x["dO"], x["dS_out"], x["dz_out"])
    b = oracle.bwd_chunked(x["q"], x["k"], x["v"], x["S0"], x["z0"], x["dO"], x["dS_out"],
                           x["dz_out"], block=block)
    for u, w in zip(a, b):
        np.testing.assert_allclose(w, u, rtol=1e-10, atol=1e-10)


def test_backward_gradient_carry_threading():
    """Backward of chunk 2 hands dS0/dz0 to chunk 1 as its dS_out/dz_out; the result
    equals the backward over both chunks in one pass."""
    x = _rand(2, 30, 4, seed=16, grads=True)
    s = 13
    sl1, sl2 = slice(0, s), slice(s, None)
    full = oracle.bwd(x["q"], x["k"], x["v"], x["S0"], x["z0"], x["dO"], x["dS_out"], x["dz_out"])
    _, S1, z1 = oracle.fwd(x["q"][:, sl1], x["k"][:, sl1], x["v"][:, sl1], x["S0"], x["z0"])
    g2 = oracle.bwd(x["q"][:, sl2], x["k"][:, sl2], x["v"][:, sl2], S1, z1, x["dO"][:, sl2],
                    x["dS_out"], x["dz_out"])
    g1 = oracle.bwd(x["q"][:, sl1], x["k"][:, sl1], x["v"][:, sl1], x["S0"], x["z0"], x["dO"][:, sl1],
                    g2[3], g2[4])
    for i in range(3):
        np.testing.assert_allclose(np.concatenate([g1[i], g2[i]], axis=1), full[i], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(g1[3], full[3], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(g1[4], full[4], rtol=1e-11, atol=1e-11)


def test_backward_null_upstream_carry_grads_are_zero():
    x = _rand(2, 9, 3, seed=17, grads=True)
    a = oracle.bwd(x["q"], x["k"], x["v"], x["S0"], x["z0"], x["dO"], None, None)
    b = oracle.bwd(x["q"], x["k"], x["v"], x["S0"], x["z0"], x["dO"], np.zeros((2, 3, 3)), np.zeros((2, 3)))
    for u, w in zip(a, b):
        np.testing.assert_array_equal(u, w)
