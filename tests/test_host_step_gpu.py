"""The host-buffer step (la_chunked_step_host): host tensors in, host tensors out.

Its results must equal, bit for bit, the device API on the same inputs (it runs the same
kernels on copies), and so match the fp64 oracle within the usual tolerances."""
import pytest
import torch

import causal_linear_attention_gb300 as la
import oracle
from causal_linear_attention_gb300.inputs import make_inputs
from parity_util import check

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
EPS = 1e-6
NAMES = ("o", "S_out", "z_out", "dq", "dk", "dv", "dS0", "dz0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    la.build()
    oracle.build()
    yield


def host_outputs(x, pinned, carries=True):
    G, C, D = x.q.shape
    mk = lambda *shape, dt: (torch.empty(*shape, dtype=dt, pin_memory=pinned))
    o, dq, dk, dv = (mk(G, C, D, dt=x.q.dtype) for _ in range(4))
    if carries:
        return (o, mk(G, D, D, dt=torch.float32), mk(G, D, dt=torch.float32), dq, dk, dv,
                mk(G, D, D, dt=torch.float32), mk(G, D, dt=torch.float32))
    return (o, None, None, dq, dk, dv, None, None)


def run_host(x, block, pinned, carries=True):
    G, C, D = x.q.shape
    xin = x
    if pinned:
        xin = type(x)(**{k: (None if t is None else t.pin_memory()) for k, t in x.__dict__.items()})
    out = host_outputs(x, pinned, carries)
    ws = la.step_workspace(G, C, D, x.q.dtype, DEV)
    s = torch.cuda.Stream(device=DEV)
    la.chunked_step_host(xin.q, xin.k, xin.v, xin.S0, xin.z0, xin.dO, xin.dS_out, xin.dz_out, out=out,
                         workspace=ws, block=block, eps=EPS, stream=s)
    s.synchronize()
    return out


def run_device(x, block):
    d = x.to(DEV)
    f = la.chunked_fwd(d.q, d.k, d.v, d.S0, d.z0, block=block, eps=EPS)
    b = la.chunked_bwd(d.q, d.k, d.v, d.S0, d.z0, d.dO, d.dS_out, d.dz_out, block=block, eps=EPS)
    torch.cuda.synchronize()
    return tuple(t.cpu() for t in f + b)


@pytest.mark.parametrize("G,C,D,dtype,block", [(160, 128, 64, "bf16", 64), (6, 200, 64, "bf16", 64),
                                               (4, 130, 128, "bf16", 128), (3, 100, 64, "f32", 64)])
def test_host_step_equals_device_api_and_oracle(G, C, D, dtype, block):
    x = make_inputs(G, C, D, dtype=dtype, seed=G + C, grads=True)
    got = run_host(x, block, pinned=True)
    dev = run_device(x, block)
    for n, a, b in zip(NAMES, got, dev):
        assert torch.equal(a, b), n
    fo = oracle.fwd(x.q, x.k, x.v, x.S0, x.z0, eps=EPS)
    bo = oracle.bwd(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, eps=EPS)
    check(got[:3], fo, dtype, NAMES[:3])
    check(got[3:], bo, dtype, NAMES[3:])


def test_host_step_pageable_memory_and_absent_carries():
    x = make_inputs(8, 128, 64, dtype="bf16", seed=3, carry=False, grads=True)
    x.dS_out = x.dz_out = None
    got = run_host(x, 64, pinned=False, carries=False)
    assert all(got[i] is None for i in (1, 2, 6, 7))
    fo = oracle.fwd(x.q, x.k, x.v, None, None, eps=EPS)
    bo = oracle.bwd(x.q, x.k, x.v, None, None, x.dO, None, None, eps=EPS)
    check((got[0],), (fo[0],), "bf16", ("o",))
    check(got[3:6], bo[:3], "bf16", ("dq", "dk", "dv"))


def test_host_step_mixed_memory_kinds():
    """Page-locked inputs with pageable outputs, and a page-locked input that is not 16-byte
    aligned: each direction takes the kernel copy only when all of its host tensors allow
    it, and the results are the same either way."""
    x = make_inputs(7, 96, 64, dtype="bf16", seed=6, grads=True)
    ref = run_device(x, 64)
    pin = {k: t.pin_memory() for k, t in x.__dict__.items()}
    ws = la.step_workspace(7, 96, 64, torch.bfloat16, DEV)
    s = torch.cuda.Stream(device=DEV)
    out = host_outputs(x, False)
    la.chunked_step_host(pin["q"], pin["k"], pin["v"], pin["S0"], pin["z0"], pin["dO"], pin["dS_out"],
                         pin["dz_out"], out=out, workspace=ws, block=64, eps=EPS, stream=s)
    s.synchronize()
    for n, a, b in zip(NAMES, out, ref):
        assert torch.equal(a, b), n
    # v 8 bytes past a 16-byte boundary of a page-locked buffer
    buf = torch.empty(x.v.numel() + 4, dtype=torch.bfloat16, pin_memory=True)
    v_odd = buf[4:].view(x.v.shape)
    v_odd.copy_(x.v)
    assert v_odd.data_ptr() % 16 == 8
    out2 = host_outputs(x, True)
    la.chunked_step_host(pin["q"], pin["k"], v_odd, pin["S0"], pin["z0"], pin["dO"], pin["dS_out"],
                         pin["dz_out"], out=out2, workspace=ws, block=64, eps=EPS, stream=s)
    s.synchronize()
    for n, a, b in zip(NAMES, out2, ref):
        assert torch.equal(a, b), n


def test_copy_kernel_needs_the_whole_buffer_page_locked():
    """The SM copy reads host memory through its device mapping, so it is chosen only when the
    first AND the last byte of a buffer are page-locked with one contiguous mapping: a buffer
    registered only in part (cudaHostRegister on a sub-range) goes to cudaMemcpyAsync.  Only
    the decision is checked here; no copy runs over the partly registered buffer."""
    pinned = torch.empty(1 << 16, dtype=torch.uint8, pin_memory=True)
    assert la.la_host_copy_eligible(pinned.data_ptr(), pinned.numel()) == 1
    assert la.la_host_copy_eligible(pinned.data_ptr() + 16, pinned.numel() - 32) == 1
    assert la.la_host_copy_eligible(pinned.data_ptr() + 8, 64) == 0      # address not 16-byte aligned
    assert la.la_host_copy_eligible(pinned.data_ptr(), 24) == 0          # length not a multiple of 16
    pageable = torch.empty(1 << 20, dtype=torch.uint8)
    assert la.la_host_copy_eligible(pageable.data_ptr(), 1 << 16) == 0
    # register the first 256 KiB of a pageable (page-aligned) region only
    base = (pageable.data_ptr() + 4095) & ~4095
    rt = torch.cuda.cudart()
    assert int(rt.cudaHostRegister(base, 1 << 18, 0)) == 0
    try:
        assert la.la_host_copy_eligible(base, 1 << 18) == 1              # inside the registration
        assert la.la_host_copy_eligible(base, (1 << 18) + 4096) == 0     # runs past its end
    finally:
        assert int(rt.cudaHostUnregister(base)) == 0
    assert la.la_host_copy_eligible(base, 1 << 18) == 0


def test_host_step_in_place_carry():
    """S_out may be the S0 buffer and dS0 the dS_out buffer: the inputs are copied in first."""
    x = make_inputs(5, 128, 64, dtype="bf16", seed=4, grads=True)
    ref = run_device(x, 64)
    S, z, dS, dz = (t.clone().pin_memory() for t in (x.S0, x.z0, x.dS_out, x.dz_out))
    q, k, v, dO = (t.pin_memory() for t in (x.q, x.k, x.v, x.dO))
    out = host_outputs(x, True)
    out = (out[0], S, z, out[3], out[4], out[5], dS, dz)
    ws = la.step_workspace(5, 128, 64, torch.bfloat16, DEV)
    s = torch.cuda.Stream(device=DEV)
    la.chunked_step_host(q, k, v, S, z, dO, dS, dz, out=out, workspace=ws, block=64, eps=EPS, stream=s)
    s.synchronize()
    for n, a, b in zip(NAMES, out, ref):
        assert torch.equal(a, b), n


def test_host_step_rejects_a_small_workspace():
    x = make_inputs(2, 16, 64, dtype="bf16", seed=5, grads=True)
    out = host_outputs(x, False)
    ws = torch.empty(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(la.LAError) as e:
        la.chunked_step_host(x.q, x.k, x.v, x.S0, x.z0, x.dO, x.dS_out, x.dz_out, out=out, workspace=ws)
    assert e.value.status == 1
