"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Workloads follow the Fractus-1B attention micro-benchmark shapes (G = B * 40 groups,
C = 128 tokens, head size 64, carry active) plus wide heads and ragged chunks;
inputs are seeded and synthetic (causal_linear_attention_gb300.inputs), the same
bits go to both sides.  Metric and tolerances: tests/parity_util.py.
"""
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


def run_fwd(x, block, eps=EPS):
    d = x.to(DEV)
    out = la.chunked_fwd(d.q, d.k, d.v, d.S0, d.z0, block=block, eps=eps)
    torch.cuda.synchronize()
    return out


def run_bwd(x, block, eps=EPS):
    d = x.to(DEV)
    out = la.chunked_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=block, eps=eps)
    torch.cuda.synchronize()
    return out


def fwd_case(G, C, D, block, dtype, seed=0, carry=True):
    x = make_inputs(G, C, D, dtype=dtype, seed=seed, carry=carry)
    got = run_fwd(x, block)
    ref = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
    return check(got, ref, dtype, FWD_NAMES)


def bwd_case(G, C, D, block, dtype, seed=0, carry=True, upstream=True):
    x = make_inputs(G, C, D, dtype=dtype, seed=seed, carry=carry, grads=True)
    if not upstream:
        x.dS_out = x.dz_out = None
    got = run_bwd(x, block)
    ref = oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS)
    return check(got, ref, dtype, BWD_NAMES)


# ------------------------------------------------------------------ the five workloads

def test_tiny_fp32_forward():
    """G=8, C=128, D=64, block=64, fp32 in and out, eps=1e-6: 1e-4 on o, S_out, z_out."""
    fwd_case(8, 128, 64, 64, "f32")


def test_tiny_fp32_backward():
    bwd_case(8, 128, 64, 64, "f32")


def test_fractus1b_block_forward():
    """B=4, niv=2, H=20 -> G=160, C=128, D=64, block=64, bf16."""
    fwd_case(160, 128, 64, 64, "bf16")


def test_fractus1b_block_backward():
    """The bench step's backward at its own size and on its own inputs (rank 0's seed):
    G=160, C=128, D=64, block=64, bf16."""
    bwd_case(160, 128, 64, 64, "bf16", seed=1000)


def test_fractus1b_forward_backward_b16():
    """B=16 -> G=640, C=128, D=64, block=64, bf16 forward + backward."""
    fwd_case(640, 128, 64, 64, "bf16", seed=2)
    bwd_case(640, 128, 64, 64, "bf16", seed=2)


def test_long_stream_carry_threaded():
    """G=160, D=64, T=8192 as 64 chunks of C=128 with the carry threaded in place;
    equals one pass of the oracle over all 8192 tokens."""
    G, C, D, nchunk = 160, 128, 64, 64
    T = C * nchunk
    x = make_inputs(G, T, D, dtype="bf16", seed=3)
    ref_o, ref_S, ref_z = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
    # chunk-major copies so that each chunk is a contiguous [G, C, D] tensor
    qc, kc, vc = (t.view(G, nchunk, C, D).transpose(0, 1).contiguous().to(DEV) for t in (x.q, x.k, x.v))
    S, z = x.S0.to(DEV).clone(), x.z0.to(DEV).clone()
    o = torch.empty(nchunk, G, C, D, device=DEV, dtype=torch.bfloat16)
    for c in range(nchunk):
        la.chunked_fwd(qc[c], kc[c], vc[c], S, z, block=64, eps=EPS, o=o[c], S_out=S, z_out=z)
    torch.cuda.synchronize()
    o_full = o.transpose(0, 1).reshape(G, T, D)
    check((o_full, S, z), (ref_o, ref_S, ref_z), "bf16", FWD_NAMES)


@pytest.mark.parametrize("block", [64, 128])
def test_wide_heads_forward_backward(block):
    """G=320, C=256, D=128, bf16, block 64 and 128."""
    fwd_case(320, 256, 128, block, "bf16", seed=4)
    bwd_case(320, 256, 128, block, "bf16", seed=4)


@pytest.mark.parametrize("block", [64, 128])
def test_wide_heads_ragged_chunk(block):
    """G=320, C=200, D=128: the last block is partial (exact in-kernel tail)."""
    fwd_case(320, 200, 128, block, "bf16", seed=5)
    bwd_case(320, 200, 128, block, "bf16", seed=5)


# ------------------------------------------------------------------ shapes, tails, edge cases

SHAPES = [(D, block) for D in (64, 128) for block in (64, 128)]


@pytest.mark.parametrize("D,block", SHAPES)
@pytest.mark.parametrize("C", [1, 15, 64, 65, 127, 130, 300])
def test_bf16_shapes_and_tails(D, block, C):
    fwd_case(5, C, D, block, "bf16", seed=C)
    bwd_case(5, C, D, block, "bf16", seed=C)


FP32_SHAPES = [(64, 64), (128, 64), (64, 128), (128, 128)]


@pytest.mark.parametrize("D,block", FP32_SHAPES)
@pytest.mark.parametrize("C", [1, 33, 128, 200])
def test_fp32_forward_shapes(D, block, C):
    fwd_case(3, C, D, block, "f32", seed=C + 1)


@pytest.mark.parametrize("D,block", FP32_SHAPES)
@pytest.mark.parametrize("C", [1, 33, 128, 200])
def test_fp32_backward_shapes(D, block, C):
    bwd_case(3, C, D, block, "f32", seed=C + 2)


@pytest.mark.parametrize("D,block", FP32_SHAPES)
def test_fp32_backward_longest_chunk(D, block):
    """The fp32 backward keeps 1/den and dd of every token on chip: the largest chunk it
    accepts (la_bwd_max_c) runs and matches the oracle, one token more is refused."""
    cmax = la.la_bwd_max_c(D, block, la.LA_F32)
    assert cmax >= 1000
    bwd_case(1, cmax, D, block, "f32", seed=D + block)
    x = make_inputs(1, cmax + 1, D, dtype="f32", seed=1, grads=True).to(DEV)
    with pytest.raises(la.LAError) as e:
        la.chunked_bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, block=block, eps=EPS)
    assert e.value.status == 2


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_zero_carry_and_no_upstream_carry_grad(dtype):
    fwd_case(4, 100, 64, 64, dtype, seed=7, carry=False)
    bwd_case(4, 100, 64, 64, dtype, seed=7, carry=False, upstream=False)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_chunk_passes_carry_through(dtype):
    x = make_inputs(3, 0, 64, dtype=dtype, seed=8, grads=True)
    o, S, z = run_fwd(x, 64)
    assert o.shape == (3, 0, 64)
    assert torch.equal(S.cpu(), x.S0) and torch.equal(z.cpu(), x.z0)
    g = run_bwd(x, 64)
    assert torch.equal(g[3].cpu(), x.dS_out) and torch.equal(g[4].cpu(), x.dz_out)


def test_single_group_full_size_and_many_groups():
    fwd_case(1, 128, 64, 64, "bf16", seed=9)
    fwd_case(1000, 64, 64, 64, "bf16", seed=10)


def test_results_are_deterministic():
    x = make_inputs(64, 200, 64, dtype="bf16", seed=11, grads=True)
    a = run_fwd(x, 64) + run_bwd(x, 64)
    b = run_fwd(x, 64) + run_bwd(x, 64)
    for u, w in zip(a, b):
        assert torch.equal(u, w)


def test_in_place_carry_and_carry_grad():
    x = make_inputs(6, 96, 64, dtype="bf16", seed=12, grads=True)
    ref = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
    d = x.to(DEV)
    S, z = d.S0.clone(), d.z0.clone()
    o, S2, z2 = la.chunked_fwd(d.q, d.k, d.v, S, z, block=64, eps=EPS, S_out=S, z_out=z)
    assert S2.data_ptr() == S.data_ptr()
    # the backward reads the ORIGINAL carry
    dS, dz = d.dS_out.clone(), d.dz_out.clone()
    out = (torch.empty_like(d.q), torch.empty_like(d.q), torch.empty_like(d.q), dS, dz)
    g = la.chunked_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, dS, dz, block=64, eps=EPS, out=out)
    torch.cuda.synchronize()
    check((o, S, z), ref, "bf16", FWD_NAMES)
    gref = oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS)
    check(g, gref, "bf16", BWD_NAMES)


def test_long_stream_single_launch():
    """The fused multi-chunk stream: G=160, D=64, T=8192 tokens in ONE forward launch (the
    carry stays on chip from tile to tile), against one oracle pass over all 8192 tokens."""
    fwd_case(160, 8192, 64, 64, "bf16", seed=3)


@pytest.mark.parametrize("G,C", [(8, 1024), (4, 1333)])
def test_wide_heads_long_chunk_forward(G, C):
    """Head size 128, many 128-token tiles in one launch (C = 1333 ends on a ragged tile)."""
    fwd_case(G, C, 128, 64, "bf16", seed=G + C)


@pytest.mark.parametrize("D,C", [(64, 128), (64, 300), (128, 200)])
def test_bf16_block_size_is_the_same_tiling(D, C):
    """The bf16 tensor-core kernels tile by 128 tokens whatever `block` is (the result is the
    same function of the inputs for every block size; only the rounding could differ, and
    here it does not): block 64 and block 128 give bit-identical outputs and gradients."""
    x = make_inputs(8, C, D, dtype="bf16", seed=D + C, grads=True)
    for u, w in zip(run_fwd(x, 64), run_fwd(x, 128)):
        assert torch.equal(u, w)
    for u, w in zip(run_bwd(x, 64), run_bwd(x, 128)):
        assert torch.equal(u, w)


def test_block_size_changes_only_rounding():
    x = make_inputs(16, 256, 64, dtype="f32", seed=13)
    a = run_fwd(x, 64)
    b = run_fwd(x, 128)
    for u, w in zip(a, b):
        assert max_rel(u, w) < 1e-5


def test_gpu_rejects_bad_arguments_without_launching():
    x = make_inputs(2, 16, 64, dtype="bf16", seed=14).to(DEV)
    o = torch.empty_like(x.q)
    with pytest.raises(la.LAError) as e:
        la.la_chunked_fwd(x.q, x.k, x.v, None, None, x.q, None, None, 2, 16, 64, 64, la.LA_BF16, EPS)
    assert e.value.status == 1
    with pytest.raises(la.LAError) as e:
        la.la_chunked_fwd(x.q, x.k, x.v, None, None, o, None, None, 2, 16, 96, 64, la.LA_BF16, EPS)
    assert e.value.status == 2
    limit = la.la_bwd_max_c(64, 64, la.LA_BF16)
    assert limit >= 4096
    with pytest.raises(la.LAError) as e:
        la.la_chunked_bwd(x.q, x.k, x.v, None, None, x.q, None, None, o, torch.empty_like(o),
                          torch.empty_like(o), None, None, 2, limit + 1, 64, 64, la.LA_BF16, EPS)
    assert e.value.status in (1, 2)
    torch.cuda.synchronize()


@pytest.mark.parametrize("C", [128, 300])
def test_backward_without_carry_gradient_outputs(C):
    """dS0 = dz0 = NULL skips those outputs; dq, dk, dv are unchanged."""
    x = make_inputs(5, C, 64, dtype="bf16", seed=15, grads=True)
    d = x.to(DEV)
    out = (torch.empty_like(d.q), torch.empty_like(d.q), torch.empty_like(d.q), None, None)
    got = la.chunked_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=64, eps=EPS, out=out)
    torch.cuda.synchronize()
    assert got[3] is None and got[4] is None
    ref = oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS)
    check(got[:3], ref[:3], "bf16", BWD_NAMES[:3])


@pytest.mark.parametrize("G,C,D", [(2, 5000, 128), (2, 17000, 64)])
def test_long_chunk_backward(G, C, D):
    """bf16 backward of chunks longer than any on-chip per-token buffer would allow
    (the kernel parks 1/den and dd in the dk rows between its passes)."""
    assert la.la_bwd_max_c(D, 64, la.LA_BF16) >= C
    bwd_case(G, C, D, 64, "bf16", seed=C)


def test_bounded_wait_gives_up_and_the_device_stays_usable():
    """Failure detection without a fault: a wait nothing satisfies gives up after its
    bound (1 ms here), the library reports it, and the next calls run normally."""
    assert la.la_device_status() == 0
    assert la.la_selftest_bounded_wait(1000) == 4  # LA_ERR_TIMEOUT, as it must
    assert la.la_device_status() == 0              # the self-test leaves the device word alone
    fwd_case(4, 128, 64, 64, "bf16", seed=21)
    assert la.la_device_status() == 0


@pytest.mark.parametrize("G,C,D", [(2, 4096, 64), (8, 1000, 64), (1, 300, 64), (3, 2048, 64),
                                   (2, 4096, 128), (8, 1000, 128), (1, 300, 128), (1, 8192, 128), (3, 2000, 128),
                                   (1, 5000, 64), (1, 12800, 128), (8, 8192, 128)])
def test_chunk_parallel_forward(G, C, D):
    """la_chunked_fwd_split (pieces on separate CTAs, carries from a prefix over the
    pieces' sums) matches the oracle, and the sequential kernel within the bf16 bounds."""
    x = make_inputs(G, C, D, dtype="bf16", seed=G * C + D, carry=True)
    ws = la.la_fwd_split_workspace_bytes(G, C, D, la.LA_BF16)
    assert ws > 0 and ws % (4 * (D * D + D)) == 0 and ws // (4 * (D * D + D)) % G == 0
    d = x.to(DEV)
    got = la.chunked_fwd_split(d.q, d.k, d.v, d.S0, d.z0, block=64, eps=EPS)
    seq = la.chunked_fwd(d.q, d.k, d.v, d.S0, d.z0, block=64, eps=EPS)
    torch.cuda.synchronize()
    ref = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
    check(got, ref, "bf16", FWD_NAMES)
    # the split sums each piece's k v^T and then prefixes the pieces: the carry's fp32 sums
    # are grouped differently from the sequential kernel's, by more as the chunk grows
    # (1.7e-5 at 12,800 tokens; 1e-2 is the carry's bound against the oracle)
    for a, b, n in zip(got, seq, FWD_NAMES):
        assert max_rel(a, b.cpu().double().numpy()) < (2e-2 if n == "o" else 5e-5), n


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("C", [129, 257, 1025])
def test_chunk_parallel_one_token_past_a_tile(D, C):
    """Chunks one token past a tile boundary: the last piece of each group holds a single
    token (forward and backward split, one group and three)."""
    for G in (1, 3):
        x = make_inputs(G, C, D, dtype="bf16", seed=C + D + G, carry=True, grads=True)
        assert la.la_fwd_split_workspace_bytes(G, C, D, la.LA_BF16) > 0
        assert la.la_bwd_split_workspace_bytes(G, C, D, la.LA_BF16) > 0
        d = x.to(DEV)
        fwd = la.chunked_fwd_split(d.q, d.k, d.v, d.S0, d.z0, block=64, eps=EPS)
        bwd = la.chunked_bwd_split(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=64, eps=EPS)
        torch.cuda.synchronize()
        assert la.la_device_status() == 0
        check(fwd, oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS), "bf16", FWD_NAMES)
        check(bwd, oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS), "bf16", BWD_NAMES)


def test_chunk_parallel_forward_falls_back_and_threads_carry_in_place():
    # many groups: no split, no workspace needed; in-place carry threading still works
    x = make_inputs(300, 256, 64, dtype="bf16", seed=5, carry=True)
    assert la.la_fwd_split_workspace_bytes(300, 256, 64, la.LA_BF16) == 0
    d = x.to(DEV)
    S, z = d.S0.clone(), d.z0.clone()
    got = la.chunked_fwd_split(d.q, d.k, d.v, S, z, block=64, eps=EPS, S_out=S, z_out=z)
    torch.cuda.synchronize()
    check(got, oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS), "bf16", FWD_NAMES)
    # a split with in-place carry: the scan reads S0 before the last piece writes S_out
    for D in (64, 128):
        x = make_inputs(2, 2000, D, dtype="bf16", seed=6, carry=True)
        d = x.to(DEV)
        S, z = d.S0.clone(), d.z0.clone()
        got = la.chunked_fwd_split(d.q, d.k, d.v, S, z, block=64, eps=EPS, S_out=S, z_out=z)
        torch.cuda.synchronize()
        check(got, oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS), "bf16", FWD_NAMES)


@pytest.mark.parametrize("G,C,D", [(2, 4096, 64), (8, 1000, 64), (1, 300, 64), (3, 2048, 64), (1, 16384, 64),
                                   (2, 4096, 128), (8, 1000, 128), (1, 300, 128), (3, 2000, 128), (1, 8192, 128),
                                   (1, 5000, 64), (1, 12800, 128), (8, 8192, 128)])
def test_chunk_parallel_backward(G, C, D):
    """la_chunked_bwd_split (forward carries from a prefix over the pieces, carry gradients
    from a reverse prefix) matches the oracle, and the sequential kernel within the bf16
    bounds."""
    x = make_inputs(G, C, D, dtype="bf16", seed=G * C + 1 + D, carry=True, grads=True)
    ws = la.la_bwd_split_workspace_bytes(G, C, D, la.LA_BF16)
    assert ws > 0 and ws % (8 * (D * D + D)) == 0
    d = x.to(DEV)
    got = la.chunked_bwd_split(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=64, eps=EPS)
    seq = la.chunked_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=64, eps=EPS)
    torch.cuda.synchronize()
    assert la.la_device_status() == 0
    ref = oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS)
    check(got, ref, "bf16", BWD_NAMES)
    for a, b, n in zip(got, seq, BWD_NAMES):
        assert max_rel(a, b.cpu().double().numpy()) < (2e-2 if n in ("dq", "dk", "dv") else 1e-4), n


@pytest.mark.parametrize("D", [64, 128])
def test_chunk_parallel_backward_carry_cases(D):
    # no upstream carry gradient, no carry
    x = make_inputs(2, 1500, D, dtype="bf16", seed=31, carry=False, grads=True)
    x.dS_out = x.dz_out = None
    d = x.to(DEV)
    got = la.chunked_bwd_split(d.q, d.k, d.v, None, None, d.dO, None, None, block=64, eps=EPS)
    torch.cuda.synchronize()
    check(got, oracle.bwd(x.q, x.k, x.v, None, None, x.dO, None, None, eps=EPS), "bf16", BWD_NAMES)
    # in place: dS0 over dS_out and dz0 over dz_out (the reverse scan reads each element
    # before it writes it)
    x = make_inputs(2, 2000, D, dtype="bf16", seed=32, carry=True, grads=True)
    d = x.to(DEV)
    dS, dz = d.dS_out.clone(), d.dz_out.clone()
    out = (torch.empty_like(d.q), torch.empty_like(d.q), torch.empty_like(d.q), dS, dz)
    got = la.chunked_bwd_split(d.q, d.k, d.v, d.S0, d.z0, d.dO, dS, dz, block=64, eps=EPS, out=out)
    torch.cuda.synchronize()
    check(got, oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS), "bf16", BWD_NAMES)
    # dS0 = dz0 = NULL: skipped
    out = (torch.empty_like(d.q), torch.empty_like(d.q), torch.empty_like(d.q), None, None)
    got = la.chunked_bwd_split(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=64, eps=EPS, out=out)
    torch.cuda.synchronize()
    ref = oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS)
    check(got[:3], ref[:3], "bf16", BWD_NAMES[:3])


def test_chunk_parallel_backward_falls_back():
    """Enough groups to fill the GPU (or one tile per chunk): no split, no workspace, the
    ordinary backward."""
    for G, C in ((300, 256), (4, 128)):
        assert la.la_bwd_split_workspace_bytes(G, C, 64, la.LA_BF16) == 0
        x = make_inputs(G, C, 64, dtype="bf16", seed=G + C, carry=True, grads=True)
        d = x.to(DEV)
        got = la.chunked_bwd_split(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=64, eps=EPS)
        torch.cuda.synchronize()
        check(got, oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS), "bf16", BWD_NAMES)
