"""GPU parity of the chunked cross-entropy over a tied head (la_ce_fwd / la_ce_bwd)
against the fp64 oracle (oracle/ce.py), through the C ABI.  Shapes: small ones with
ragged chunks, and the page's head (N = 512 tokens, V = 50257, d = 1280) whole and in
chunks of 128.  Inputs from the shared seeded generator; the oracle decodes the same
bf16 bits.  Tolerances (a reading: the page states none): loss and lse 1e-4 relative
(fp32 accumulation over d), dh and dW 2e-2 normwise (the gradient rows are rounded to
bf16 before the two GEMMs)."""
import numpy as np
import pytest
import torch

import causal_linear_attention_gb300 as la
from causal_linear_attention_gb300.inputs import CE_SHAPE, make_ce_inputs
from oracle import ce
from parity_util import max_rel

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    la.build()
    yield


def run(N, V, d, chunk, seed, dloss=1.0):
    h, W, y = make_ce_inputs(N, V, d, seed)
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    ws = la.ce_workspace(N, V, d, chunk, DEV)
    loss, lse = la.ce_fwd(hd, Wd, yd, ce_chunk=chunk, workspace=ws)
    dh, dW = la.ce_bwd(hd, Wd, yd, lse, dloss, ce_chunk=chunk, workspace=ws)
    torch.cuda.synchronize()
    assert la.la_device_status() == 0
    return (h, W, y), (float(loss), lse.cpu().double().numpy(), dh, dW)


def check(inp, got, chunk, dloss=1.0):
    h, W, y = inp
    loss, lse, dh, dW = got
    r_loss, r_lse = ce.ce_fwd_chunked(h, W, y.numpy(), chunk)
    r_dh, r_dW = ce.ce_bwd_chunked(h, W, y.numpy(), chunk, dloss)
    assert abs(loss - r_loss) / abs(r_loss) < 1e-4
    assert max_rel(lse, r_lse) < 1e-4
    assert max_rel(dh, r_dh) < 2e-2, max_rel(dh, r_dh)
    assert max_rel(dW, r_dW) < 2e-2, max_rel(dW, r_dW)


@pytest.mark.parametrize("N,V,d,chunk", [(300, 1000, 128, 64), (300, 1000, 128, 300), (257, 4099, 64, 100),
                                         (1, 7, 64, 4), (512, 9728, 128, 512)])
def test_ce_matches_oracle(N, V, d, chunk):
    """The fused GEMM's vocabulary tile follows the waves over the SMs: on 152 SMs the
    small shapes take 192-row tiles, (512, 9728) 256-row ones, and the page's head 224
    (chunks of 512) and 192 (chunks of 128)."""
    inp, got = run(N, V, d, chunk, seed=N + V)
    check(inp, got, chunk)


@pytest.mark.parametrize("chunk", [512, 128])
def test_ce_fractus1b_head(chunk):
    """The page's head: 512 tokens, 50257-token vocabulary, d = 1280."""
    inp, got = run(CE_SHAPE["N"], CE_SHAPE["V"], CE_SHAPE["d"], chunk, seed=3)
    check(inp, got, chunk)


def test_ce_chunking_and_dloss():
    """Chunk size changes only rounding; dloss scales both gradients."""
    _, a = run(200, 3000, 64, 200, seed=5)
    _, b = run(200, 3000, 64, 37, seed=5, dloss=0.5)
    assert abs(a[0] - b[0]) < 1e-5 * abs(a[0])
    assert max_rel(b[2].float() * 2, a[2]) < 2e-2
    assert max_rel(b[3] * 2, a[3]) < 1e-2


def test_ce_is_deterministic():
    _, a = run(300, 2000, 128, 128, seed=6)
    _, b = run(300, 2000, 128, 128, seed=6)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])


def test_ce_empty_batch():
    h = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(10, 64, device=DEV).to(torch.bfloat16)
    y = torch.empty(0, dtype=torch.int32, device=DEV)
    loss, lse = la.ce_fwd(h, W, y, ce_chunk=8, workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    dh, dW = la.ce_bwd(h, W, y, lse, ce_chunk=8, workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    assert float(loss) == 0.0 and dh.numel() == 0 and not dW.any()


@pytest.mark.parametrize("N,V,d,chunk", [(200, 700, 192, 77), (129, 3000, 320, 129)])
def test_ce_gemm_tails(N, V, d, chunk):
    """The backward's GEMMs at widths that leave part of a 256-column tile empty (d = 192,
    320), a vocabulary that is not a multiple of 64 and chunks that are not a multiple of
    the 128-token tile."""
    inp, got = run(N, V, d, chunk, seed=N + d)
    check(inp, got, chunk)


def test_ce_out_of_range_target_is_reported():
    """A target outside [0, V): that row's loss is NaN (the kernel reads nothing outside
    the row) and la_device_status reports LA_ERR_DEVICE; the next calls are clean."""
    h, W, y = make_ce_inputs(8, 50, 64, seed=7)
    y[3] = 50
    hd, Wd, yd = h.to(DEV), W.to(DEV), y.to(DEV)
    loss, _ = la.ce_fwd(hd, Wd, yd, ce_chunk=8)
    torch.cuda.synchronize()
    assert np.isnan(float(loss))
    assert la.la_device_status(1) == 5  # LA_ERR_DEVICE, and clear it
    assert la.la_device_status() == 0
    inp, got = run(8, 50, 64, 8, seed=7)
    check(inp, got, 8)
