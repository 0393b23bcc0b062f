"""The C-ABI library builds, loads and exports every symbol include/la.h declares;
host-side argument checks reject bad calls before anything touches a GPU."""
import os
import re
import shutil

import pytest

import causal_linear_attention_gb300 as la
from causal_linear_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "la.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not available")


@pytest.fixture(scope="module")
def L():
    la.build()
    return la.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(["la_chunked_fwd", "la_chunked_bwd", "la_fwd_split_workspace_bytes",
                                           "la_chunked_fwd_split", "la_chunked_fwd_split_static",
                                           "la_bwd_split_workspace_bytes", "la_chunked_bwd_split",
                                           "la_cumsum_fwd", "la_cumsum_bwd_workspace_bytes", "la_cumsum_bwd",
                                           "la_ce_workspace_bytes", "la_ce_fwd", "la_ce_bwd",
                                           "la_step_workspace_bytes",
                                           "la_chunked_step_host", "la_host_copy_eligible", "la_bwd_max_c",
                                           "la_device_status",
                                           "la_selftest_bounded_wait", "la_status_string", "la_version"])


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(_lib.EXPORTS) == set(declared_functions())


def test_status_strings_and_version(L):
    assert la.la_version() == 100
    for s in range(6):
        assert len(la.la_status_string(s)) > 0


# Fake, 16-byte aligned "device" addresses.  Every call below must fail its host-side
# checks (so nothing is ever launched on them, with or without a GPU present).
A = 0x10000


def fwd(**kw):
    args = dict(q=A, k=A + 0x100000, v=A + 0x200000, S0=None, z0=None, o=A + 0x300000, S_out=None,
                z_out=None, G=2, C=8, D=64, block=64, dtype=la.LA_BF16, eps=1e-6)
    args.update(kw)
    L = la.lib()
    return L.la_chunked_fwd(args["q"], args["k"], args["v"], args["S0"], args["z0"], args["o"],
                            args["S_out"], args["z_out"], args["G"], args["C"], args["D"], args["block"],
                            args["dtype"], args["eps"], None)


def bwd(**kw):
    base = {n: A + i * 0x100000 for i, n in enumerate(("q", "k", "v", "dO", "dq", "dk", "dv"))}
    args = dict(base, S0=None, z0=None, dS_out=None, dz_out=None, dS0=None, dz0=None, G=2, C=8, D=64,
                block=64, dtype=la.LA_BF16, eps=1e-6)
    args.update(kw)
    L = la.lib()
    return L.la_chunked_bwd(args["q"], args["k"], args["v"], args["S0"], args["z0"], args["dO"],
                            args["dS_out"], args["dz_out"], args["dq"], args["dk"], args["dv"], args["dS0"],
                            args["dz0"], args["G"], args["C"], args["D"], args["block"], args["dtype"],
                            args["eps"], None)


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("kw,status", [
    (dict(G=-1), INVALID), (dict(C=-5), INVALID), (dict(q=None), INVALID), (dict(o=None), INVALID),
    (dict(q=A + 4), INVALID), (dict(eps=float("nan")), INVALID), (dict(eps=float("inf")), INVALID),
    (dict(D=32), UNSUPPORTED), (dict(D=96), UNSUPPORTED), (dict(block=32), UNSUPPORTED),
    (dict(dtype=7), UNSUPPORTED),
    (dict(o=A), INVALID),                       # output overlaps q
    (dict(S0=A + 0x400000, S_out=A + 0x400010), INVALID),  # partial overlap of the carry
    (dict(z_out=A + 0x300000), INVALID),        # z_out inside o
])
def test_forward_argument_checks(L, kw, status):
    assert fwd(**kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(G=-1), INVALID), (dict(dq=None), INVALID), (dict(dO=None), INVALID), (dict(dk=A + 8), INVALID),
    (dict(D=48), UNSUPPORTED), (dict(block=256), UNSUPPORTED),
    (dict(dq=A), INVALID),                      # dq overlaps q
    (dict(dk=A + 0x400000, dv=A + 0x400000), INVALID),  # two outputs share memory
    (dict(dS_out=A + 0x800000, dS0=A + 0x800040), INVALID),
])
def test_backward_argument_checks(L, kw, status):
    assert bwd(**kw) == status


def test_empty_problems_are_accepted_without_a_launch(L):
    assert fwd(G=0) == 0
    assert bwd(G=0) == 0
    # G = 0 with NULL buffers is fine: there is nothing to read or write
    assert fwd(G=0, q=None, k=None, v=None, o=None) == 0


def test_raw_binding_raises_on_error(L):
    with pytest.raises(la.LAError) as e:
        la.la_chunked_fwd(A, A, A, None, None, A, None, None, 1, 8, 64, 64, la.LA_BF16, 1e-6)
    assert e.value.status == 1  # o overlaps the inputs: rejected before any CUDA call


@pytest.mark.parametrize("G,C,D,dtype", [(160, 128, 64, 1), (3, 200, 128, 1), (8, 128, 64, 0), (1, 1, 64, 1),
                                         (0, 128, 64, 1), (5, 0, 64, 0)])
def test_step_workspace_bytes_closed_form(L, G, C, D, dtype):
    """Sixteen slots (8 token tensors, 4 D x D carries, 4 length-D carries), each
    rounded up to 256 bytes."""
    e = 4 if dtype == 0 else 2
    r = lambda n: (n + 255) // 256 * 256
    want = 8 * r(G * C * D * e) + 4 * r(G * D * D * 4) + 4 * r(G * D * 4)
    assert la.la_step_workspace_bytes(G, C, D, dtype) == want


def test_ce_needs_d_a_multiple_of_64(L):
    """The cross-entropy runs on the tensor-core kernels, which take d in 64-wide slices: any
    other d gets no workspace size and is refused before any CUDA call."""
    assert la.la_ce_workspace_bytes(8, 50, 64, 8) > 0
    assert la.la_ce_workspace_bytes(8, 50, 96, 8) == 0
    A = 0x20000000
    assert L.la_ce_fwd(A, A + 0x100000, A + 0x200000, 8, 50, 96, 8, A + 0x300000, A + 0x300100, A + 0x400000,
                       1 << 24, None) == UNSUPPORTED


def test_step_workspace_bytes_rejects_bad_shapes(L):
    assert la.la_step_workspace_bytes(2, 8, 96, 1) == 0
    assert la.la_step_workspace_bytes(-1, 8, 64, 1) == 0
    assert la.la_step_workspace_bytes(2, 8, 64, 9) == 0


# Host-buffer step: fake host pointers; every call below must fail its argument checks
# before any copy is enqueued (G = 0 returns before touching anything).
H = 0x7F0000000000


def step(**kw):
    names = ("q", "k", "v", "S0", "z0", "dO", "dS_out", "dz_out", "o", "S_out", "z_out", "dq", "dk", "dv", "dS0",
             "dz0")
    args = {n: H + i * 0x1000000 for i, n in enumerate(names)}
    for n in ("S0", "z0", "dS_out", "dz_out", "S_out", "z_out", "dS0", "dz0"):
        args[n] = None
    args.update(workspace=0x20000000, workspace_bytes=1 << 30, G=2, C=8, D=64, block=64, dtype=la.LA_BF16,
                eps=1e-6)
    args.update(kw)
    L = la.lib()
    return L.la_chunked_step_host(*(args[n] for n in names), args["workspace"], args["workspace_bytes"],
                                  args["G"], args["C"], args["D"], args["block"], args["dtype"], args["eps"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), INVALID), (dict(dO=None), INVALID), (dict(o=None), INVALID), (dict(dv=None), INVALID),
    (dict(workspace=None), INVALID), (dict(workspace_bytes=1000), INVALID), (dict(workspace=0x20000010), INVALID),
    (dict(o=H), INVALID),                                   # output overlaps q
    (dict(dq=H + 0x8000000 + 0x100), INVALID),             # dq overlaps o
    (dict(S0=H + 0x30000000, S_out=H + 0x30000040), INVALID),  # partial overlap of the carry
    (dict(D=96), UNSUPPORTED), (dict(dtype=5), UNSUPPORTED), (dict(G=-3), INVALID),
])
def test_host_step_argument_checks(L, kw, status):
    assert step(**kw) == status


def test_selftest_rejects_out_of_range_waits_before_any_cuda_call(L):
    assert la.la_selftest_bounded_wait(0) == INVALID
    assert la.la_selftest_bounded_wait(2_000_000) == INVALID


def test_host_step_empty_problem_is_accepted_without_copies(L):
    assert step(G=0) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(G=-1), INVALID), (dict(q=None), INVALID), (dict(o=None), INVALID), (dict(q=A + 4), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(o=A), INVALID),
])
def test_split_forward_entry_points_check_arguments_first(L, kw, status):
    """Both chunk-parallel entry points run the forward's checks before any CUDA call."""
    args = dict(q=A, k=A + 0x100000, v=A + 0x200000, S0=None, z0=None, o=A + 0x300000, S_out=None,
                z_out=None, G=2, C=8, D=64, block=64, dtype=la.LA_BF16, eps=1e-6)
    args.update(kw)
    head = [args[n] for n in ("q", "k", "v", "S0", "z0", "o", "S_out", "z_out")]
    tail = [args[n] for n in ("G", "C", "D", "block", "dtype", "eps")]
    assert L.la_chunked_fwd_split(*head, *tail, None, 0, None) == status
    assert L.la_chunked_fwd_split_static(*head, *tail, None) == status


@pytest.mark.parametrize("kw,status", [
    (dict(G=-1), INVALID), (dict(dq=None), INVALID), (dict(dO=None), INVALID), (dict(dk=A + 8), INVALID),
    (dict(D=48), UNSUPPORTED), (dict(dq=A), INVALID), (dict(dk=A + 0x400000, dv=A + 0x400000), INVALID),
])
def test_split_backward_checks_arguments_first(L, kw, status):
    """The chunk-parallel backward runs the backward's checks before any CUDA call."""
    base = {n: A + i * 0x100000 for i, n in enumerate(("q", "k", "v", "dO", "dq", "dk", "dv"))}
    args = dict(base, S0=None, z0=None, dS_out=None, dz_out=None, dS0=None, dz0=None, G=2, C=8, D=64,
                block=64, dtype=la.LA_BF16, eps=1e-6)
    args.update(kw)
    names = ("q", "k", "v", "S0", "z0", "dO", "dS_out", "dz_out", "dq", "dk", "dv", "dS0", "dz0", "G", "C", "D",
             "block", "dtype", "eps")
    assert L.la_chunked_bwd_split(*(args[n] for n in names), None, 0, None) == status


def test_split_workspace_is_zero_where_no_split_applies(L):
    """No split (so no workspace) for fp32 or chunks of one tile; the calls make no kernel
    launch to decide that."""
    for f in (la.la_fwd_split_workspace_bytes, la.la_bwd_split_workspace_bytes):
        for D in (64, 128):
            assert f(2, 4096, D, la.LA_F32) == 0
            assert f(2, 128, D, la.LA_BF16) == 0
            assert f(-1, 4096, D, la.LA_BF16) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(G=-1), INVALID), (dict(q=None), INVALID), (dict(o=None), INVALID), (dict(q=A + 4), INVALID),
    (dict(D=96), UNSUPPORTED), (dict(dtype=7), UNSUPPORTED), (dict(o=A), INVALID), (dict(eps=float("nan")), INVALID),
])
def test_cumsum_forward_checks_arguments_first(L, kw, status):
    args = dict(q=A, k=A + 0x100000, v=A + 0x200000, S0=None, z0=None, o=A + 0x300000, S_out=None,
                z_out=None, G=2, C=8, D=64, dtype=la.LA_BF16, eps=1e-6)
    args.update(kw)
    names = ("q", "k", "v", "S0", "z0", "o", "S_out", "z_out", "G", "C", "D", "dtype", "eps")
    assert L.la_cumsum_fwd(*(args[n] for n in names), None) == status


@pytest.mark.parametrize("kw,status", [
    (dict(G=-1), INVALID), (dict(dq=None), INVALID), (dict(dk=A + 8), INVALID), (dict(D=48), UNSUPPORTED),
    (dict(dq=A), INVALID), (dict(workspace=None), INVALID), (dict(workspace_bytes=64), INVALID),
    (dict(workspace=0x20000008), INVALID), (dict(workspace=A), INVALID),  # misaligned; overlaps q
    (dict(G=715827883, C=0), UNSUPPORTED),  # three CTAs per group would overflow the grid
])
def test_cumsum_backward_checks_arguments_first(L, kw, status):
    base = {n: A + i * 0x100000 for i, n in enumerate(("q", "k", "v", "dO", "dq", "dk", "dv"))}
    args = dict(base, S0=None, z0=None, dS_out=None, dz_out=None, dS0=None, dz0=None, G=2, C=8, D=64,
                dtype=la.LA_BF16, eps=1e-6, workspace=0x20000000, workspace_bytes=1 << 20)
    args.update(kw)
    names = ("q", "k", "v", "S0", "z0", "dO", "dS_out", "dz_out", "dq", "dk", "dv", "dS0", "dz0", "G", "C", "D",
             "dtype", "eps", "workspace", "workspace_bytes")
    assert L.la_cumsum_bwd(*(args[n] for n in names), None) == status


def test_cumsum_workspace_bytes_closed_form(L):
    """Two fp32 values per token (1/den and dd), rounded up to a multiple of four, then one
    D x D fp32 copy of dS_out per group; nothing for an empty chunk."""
    for G, C, D, dt in ((160, 128, 64, 1), (3, 200, 128, 0), (0, 5, 64, 1), (4, 0, 64, 1), (3, 33, 64, 1)):
        want = 0 if C == 0 else ((2 * G * C + 3) // 4 * 4 + G * D * D) * 4
        assert la.la_cumsum_bwd_workspace_bytes(G, C, D, dt) == want
    assert la.la_cumsum_bwd_workspace_bytes(2, 8, 96, 1) == 0


def test_ce_workspace_bytes_closed_form(L):
    """The chunk's vocabulary-major bf16 gradient (the chunk padded to 32 tokens), N floats,
    two [tiles][chunk] partial arrays (a slot per tile of the narrowest vocabulary tile, 192
    rows), the chunk's target logits and 8 fp32 [chunk][d] partial sums of dh, each rounded
    up to 256 bytes; the chunk is at most N tokens; d must be a multiple of 64."""
    r = lambda n: (n + 255) // 256 * 256
    for N, V, d, cc in ((512, 50257, 1280, 512), (512, 50257, 1280, 128), (300, 1000, 128, 1000), (1, 7, 64, 4)):
        cs, ns = (min(cc, N) + 31) // 32 * 32, (V + 191) // 192
        want = r(V * cs * 2) + r(N * 4) + 2 * r(ns * cs * 4) + r(cs * 4) + r(8 * cs * d * 4)
        assert la.la_ce_workspace_bytes(N, V, d, cc) == want
    assert la.la_ce_workspace_bytes(-1, 5, 64, 5) == 0
    assert la.la_ce_workspace_bytes(5, 0, 64, 5) == 0
    assert la.la_ce_workspace_bytes(5, 5, 64, 0) == 0
    assert la.la_ce_workspace_bytes(5, 5, 8, 5) == 0


def ce_call(fwd=True, **kw):
    WS = 0x40000000
    args = dict(h=A, W=A + 0x100000, targets=A + 0x200000, lse=A + 0x300000, loss=A + 0x400000,
                dh=A + 0x500000, dW=A + 0x600000, N=4, V=16, d=64, ce_chunk=4, workspace=WS, workspace_bytes=1 << 30)
    args.update(kw)
    L = la.lib()
    if fwd:
        return L.la_ce_fwd(args["h"], args["W"], args["targets"], args["N"], args["V"], args["d"], args["ce_chunk"],
                           args["loss"], args["lse"], args["workspace"], args["workspace_bytes"], None)
    return L.la_ce_bwd(args["h"], args["W"], args["targets"], args["lse"], 1.0, args["N"], args["V"], args["d"],
                       args["ce_chunk"], args["dh"], args["dW"], args["workspace"], args["workspace_bytes"], None)


@pytest.mark.parametrize("fwd", [True, False])
@pytest.mark.parametrize("kw", [dict(N=-1), dict(V=0), dict(d=0), dict(ce_chunk=0), dict(h=None), dict(W=None),
                                dict(targets=None), dict(h=A + 8), dict(targets=A + 0x200002), dict(workspace=None),
                                dict(workspace=0x40000010), dict(workspace_bytes=1000), dict(workspace=A)])
def test_ce_checks_arguments_first(L, fwd, kw):
    assert ce_call(fwd, **kw) == INVALID


def test_ce_output_checks(L):
    assert ce_call(True, loss=None) == INVALID
    assert ce_call(True, lse=A) == INVALID          # lse over h
    assert ce_call(False, dh=None) == INVALID
    assert ce_call(False, dW=A + 0x100000) == INVALID  # dW over W


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.lib()
