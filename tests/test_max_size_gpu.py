"""Maximum sizes: more groups than a 32-bit element offset can address.

G = 262,400 groups of C = 128 tokens at D = 64 puts 2.15e9 elements in every [G, C, D]
tensor (4.3 GB in bf16), so group g's rows start past 2^31 elements for g >= 262,144.
The inputs are the 160 seeded groups of the Fractus-1B block repeated 1,640 times, so
every group has a small oracle: sampled groups, low and high, are checked against the
fp64 oracle and bit for bit against the group with the same inputs near the start
(each group runs alone in its CTA, so equal inputs give equal bits).  About 55 GB of
device memory."""
import pytest
import torch

import causal_linear_attention_gb300 as la
import oracle
from causal_linear_attention_gb300.inputs import make_inputs
from parity_util import check

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
EPS = 1e-6
BASE, REPS = 160, 1640
G = BASE * REPS
SAMPLES = (0, 159, 131_077, 262_143, 262_144, 262_205, G - 1)


@pytest.fixture(scope="module")
def big():
    la.build()
    oracle.build()
    if torch.cuda.mem_get_info(DEV)[0] < 80 * 2**30:
        pytest.skip("needs about 55 GB of free device memory")
    x = make_inputs(BASE, 128, 64, dtype="bf16", seed=21, carry=True, grads=True)
    rep = lambda t: t.to(DEV).repeat(REPS, *([1] * (t.dim() - 1))).contiguous()
    d = {k: rep(t) for k, t in x.__dict__.items()}
    assert d["q"].numel() > 2**31
    yield x, d
    del d
    torch.cuda.empty_cache()


def sample(t, g):
    return t[g].cpu()


def test_forward_and_backward_past_32bit_offsets(big):
    x, d = big
    o, S, z = la.chunked_fwd(d["q"], d["k"], d["v"], d["S0"], d["z0"], block=64, eps=EPS)
    grads = la.chunked_bwd(d["q"], d["k"], d["v"], d["S0"], d["z0"], d["dO"], d["dS_out"], d["dz_out"], block=64,
                           eps=EPS)
    torch.cuda.synchronize()
    assert la.la_device_status() == 0
    ref_f = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
    ref_b = oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS)
    outs = (o, S, z) + tuple(grads)
    names = ("o", "S_out", "z_out", "dq", "dk", "dv", "dS0", "dz0")
    for g in SAMPLES:
        b = g % BASE
        got = [sample(t, g) for t in outs]
        check(got[:3], [r[b] for r in ref_f], "bf16", names[:3])
        check(got[3:], [r[b] for r in ref_b], "bf16", names[3:])
        for n, a, t in zip(names, got, outs):
            assert torch.equal(a, sample(t, b)), (n, g)


def test_cumsum_form_past_32bit_offsets(big):
    x, d = big
    o, S, z = la.cumsum_fwd(d["q"], d["k"], d["v"], d["S0"], d["z0"], eps=EPS)
    torch.cuda.synchronize()
    ref = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
    for g in SAMPLES:
        b = g % BASE
        got = [sample(t, g) for t in (o, S, z)]
        check(got, [r[b] for r in ref], "bf16", ("o", "S_out", "z_out"))
        for a, t in zip(got, (o, S, z)):
            assert torch.equal(a, sample(t, b))
