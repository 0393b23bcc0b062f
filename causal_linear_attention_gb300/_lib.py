"""ctypes binding of libla.so (include/la.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  PyTorch is used
for device memory and streams.  There is no fallback: if the library is missing
or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_BUILD = os.path.join(_PKG, "_build")
LIB_PATH = os.path.join(_BUILD, "libla.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

LA_F32, LA_BF16 = 0, 1
STATUS = {0: "LA_OK", 1: "LA_ERR_INVALID", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_CUDA", 4: "LA_ERR_TIMEOUT", 5: "LA_ERR_DEVICE"}

_lib = None
_lock = threading.Lock()


class LAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def _sources():
    srcs = [os.path.join(_CSRC, f) for f in sorted(os.listdir(_CSRC)) if f.endswith((".cu", ".cuh"))]
    return srcs + [os.path.join(_INCLUDE, "la.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a into _build/libla.so (skipped when up to date)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(LIB_PATH):
        newest = max(os.path.getmtime(s) for s in _sources())
        if os.path.getmtime(LIB_PATH) >= newest:
            return LIB_PATH
    units = [os.path.join(_CSRC, f) for f in sorted(os.listdir(_CSRC)) if f.endswith(".cu")]
    objs = []
    procs = []
    for u in units:  # one process per translation unit, in parallel
        obj = os.path.join(_BUILD, os.path.basename(u)[:-3] + ".o")
        cmd = ["nvcc", ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               f"-I{_INCLUDE}", "-c", u, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((subprocess.Popen(cmd), cmd))
        objs.append(obj)
    for p, cmd in procs:
        if p.wait() != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["nvcc", ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
                    *objs, "-o", tmp], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run causal_linear_attention_gb300.build() "
                               "(nvcc, sm_103a) first; there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.la_chunked_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, F, P]
        L.la_chunked_fwd.restype = I
        L.la_chunked_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P]
        L.la_chunked_bwd.restype = I
        L.la_device_status.argtypes = [I]
        L.la_device_status.restype = I
        L.la_step_workspace_bytes.argtypes = [I, I, I, I]
        L.la_step_workspace_bytes.restype = ctypes.c_size_t
        L.la_chunked_step_host.argtypes = [P] * 17 + [ctypes.c_size_t, I, I, I, I, I, F, P]
        L.la_chunked_step_host.restype = I
        L.la_host_copy_eligible.argtypes = [P, ctypes.c_size_t]
        L.la_host_copy_eligible.restype = I
        L.la_fwd_split_workspace_bytes.argtypes = [I, I, I, I]
        L.la_fwd_split_workspace_bytes.restype = ctypes.c_size_t
        L.la_chunked_fwd_split.argtypes = [P] * 8 + [I, I, I, I, I, F, P, ctypes.c_size_t, P]
        L.la_chunked_fwd_split.restype = I
        L.la_chunked_fwd_split_static.argtypes = [P] * 8 + [I, I, I, I, I, F, P]
        L.la_chunked_fwd_split_static.restype = I
        L.la_ce_workspace_bytes.argtypes = [I, I, I, I]
        L.la_ce_workspace_bytes.restype = ctypes.c_size_t
        L.la_ce_fwd.argtypes = [P, P, P, I, I, I, I, P, P, P, ctypes.c_size_t, P]
        L.la_ce_fwd.restype = I
        L.la_ce_bwd.argtypes = [P, P, P, P, F, I, I, I, I, P, P, P, ctypes.c_size_t, P]
        L.la_ce_bwd.restype = I
        L.la_cumsum_fwd.argtypes = [P] * 8 + [I, I, I, I, F, P]
        L.la_cumsum_fwd.restype = I
        L.la_cumsum_bwd_workspace_bytes.argtypes = [I, I, I, I]
        L.la_cumsum_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.la_cumsum_bwd.argtypes = [P] * 13 + [I, I, I, I, F, P, ctypes.c_size_t, P]
        L.la_cumsum_bwd.restype = I
        L.la_bwd_split_workspace_bytes.argtypes = [I, I, I, I]
        L.la_bwd_split_workspace_bytes.restype = ctypes.c_size_t
        L.la_chunked_bwd_split.argtypes = [P] * 13 + [I, I, I, I, I, F, P, ctypes.c_size_t, P]
        L.la_chunked_bwd_split.restype = I
        L.la_selftest_bounded_wait.argtypes = [I]
        L.la_selftest_bounded_wait.restype = I
        L.la_bwd_max_c.argtypes = [I, I, I]
        L.la_bwd_max_c.restype = I
        L.la_status_string.argtypes = [I]
        L.la_status_string.restype = ctypes.c_char_p
        L.la_version.argtypes = []
        L.la_version.restype = I
        _lib = L
        return L


EXPORTS = ("la_chunked_fwd", "la_chunked_bwd", "la_fwd_split_workspace_bytes", "la_chunked_fwd_split",
           "la_chunked_fwd_split_static", "la_bwd_split_workspace_bytes", "la_chunked_bwd_split",
           "la_cumsum_fwd", "la_cumsum_bwd_workspace_bytes", "la_cumsum_bwd",
           "la_ce_workspace_bytes", "la_ce_fwd", "la_ce_bwd",
           "la_step_workspace_bytes", "la_chunked_step_host", "la_host_copy_eligible", "la_bwd_max_c",
           "la_device_status", "la_selftest_bounded_wait", "la_status_string", "la_version")


def _p(x) -> Optional[int]:
    """Pointer of a tensor / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _check(status: int):
    if status != 0:
        raise LAError(status, lib().la_status_string(status).decode())


def la_chunked_fwd(q, k, v, S0, z0, o, S_out, z_out, G: int, C: int, D: int, block: int,
                   dtype: int, eps: float, stream=None) -> None:
    """Raw C-ABI call (device pointers or tensors).  Raises LAError on a non-OK status."""
    _check(lib().la_chunked_fwd(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(o), _p(S_out), _p(z_out),
                                G, C, D, block, dtype, eps, _p(stream)))


def la_chunked_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G: int, C: int, D: int,
                   block: int, dtype: int, eps: float, stream=None) -> None:
    """Raw C-ABI call (device pointers or tensors).  Raises LAError on a non-OK status."""
    _check(lib().la_chunked_bwd(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(dO), _p(dS_out), _p(dz_out),
                                _p(dq), _p(dk), _p(dv), _p(dS0), _p(dz0), G, C, D, block, dtype, eps,
                                _p(stream)))


def la_fwd_split_workspace_bytes(G: int, C: int, D: int, dtype: int) -> int:
    return int(lib().la_fwd_split_workspace_bytes(G, C, D, dtype))


def la_chunked_fwd_split(q, k, v, S0, z0, o, S_out, z_out, G: int, C: int, D: int, block: int, dtype: int,
                         eps: float, workspace, workspace_bytes: int, stream=None) -> None:
    """Raw C-ABI call (device pointers or tensors).  Raises LAError on a non-OK status."""
    _check(lib().la_chunked_fwd_split(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(o), _p(S_out), _p(z_out), G, C, D,
                                      block, dtype, eps, _p(workspace), workspace_bytes, _p(stream)))


def la_ce_workspace_bytes(N: int, V: int, d: int, ce_chunk: int) -> int:
    return int(lib().la_ce_workspace_bytes(N, V, d, ce_chunk))


def la_ce_fwd(h, W, targets, N: int, V: int, d: int, ce_chunk: int, loss, lse, workspace, workspace_bytes: int,
              stream=None) -> None:
    """Raw C-ABI call of the chunked cross-entropy forward (device pointers or tensors)."""
    _check(lib().la_ce_fwd(_p(h), _p(W), _p(targets), N, V, d, ce_chunk, _p(loss), _p(lse), _p(workspace),
                           workspace_bytes, _p(stream)))


def la_ce_bwd(h, W, targets, lse, dloss: float, N: int, V: int, d: int, ce_chunk: int, dh, dW, workspace,
              workspace_bytes: int, stream=None) -> None:
    """Raw C-ABI call of the chunked cross-entropy backward."""
    _check(lib().la_ce_bwd(_p(h), _p(W), _p(targets), _p(lse), dloss, N, V, d, ce_chunk, _p(dh), _p(dW),
                           _p(workspace), workspace_bytes, _p(stream)))


def la_cumsum_fwd(q, k, v, S0, z0, o, S_out, z_out, G: int, C: int, D: int, dtype: int, eps: float,
                  stream=None) -> None:
    """Raw C-ABI call of the cumsum form (device pointers or tensors)."""
    _check(lib().la_cumsum_fwd(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(o), _p(S_out), _p(z_out), G, C, D, dtype, eps,
                               _p(stream)))


def la_cumsum_bwd_workspace_bytes(G: int, C: int, D: int, dtype: int) -> int:
    return int(lib().la_cumsum_bwd_workspace_bytes(G, C, D, dtype))


def la_cumsum_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G: int, C: int, D: int, dtype: int,
                  eps: float, workspace, workspace_bytes: int, stream=None) -> None:
    """Raw C-ABI call of the cumsum form's backward."""
    _check(lib().la_cumsum_bwd(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(dO), _p(dS_out), _p(dz_out), _p(dq), _p(dk),
                               _p(dv), _p(dS0), _p(dz0), G, C, D, dtype, eps, _p(workspace), workspace_bytes,
                               _p(stream)))


def la_bwd_split_workspace_bytes(G: int, C: int, D: int, dtype: int) -> int:
    return int(lib().la_bwd_split_workspace_bytes(G, C, D, dtype))


def la_chunked_bwd_split(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G: int, C: int, D: int,
                         block: int, dtype: int, eps: float, workspace, workspace_bytes: int, stream=None) -> None:
    """Raw C-ABI call (device pointers or tensors).  Raises LAError on a non-OK status."""
    _check(lib().la_chunked_bwd_split(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(dO), _p(dS_out), _p(dz_out), _p(dq),
                                      _p(dk), _p(dv), _p(dS0), _p(dz0), G, C, D, block, dtype, eps, _p(workspace),
                                      workspace_bytes, _p(stream)))


def la_chunked_fwd_split_static(q, k, v, S0, z0, o, S_out, z_out, G: int, C: int, D: int, block: int, dtype: int,
                                eps: float, stream=None) -> None:
    """Raw C-ABI call of the chunk-parallel forward that needs no workspace (module-level
    device scratch; calls on one device must not overlap in time)."""
    _check(lib().la_chunked_fwd_split_static(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(o), _p(S_out), _p(z_out), G, C,
                                             D, block, dtype, eps, _p(stream)))


def la_step_workspace_bytes(G: int, C: int, D: int, dtype: int) -> int:
    return int(lib().la_step_workspace_bytes(G, C, D, dtype))


def la_host_copy_eligible(ptr: int, nbytes: int) -> int:
    """1 when la_chunked_step_host would move this host buffer with its SM-copy kernel."""
    return int(lib().la_host_copy_eligible(ctypes.c_void_p(ptr), nbytes))


def la_chunked_step_host(q, k, v, S0, z0, dO, dS_out, dz_out, o, S_out, z_out, dq, dk, dv, dS0, dz0,
                         workspace, workspace_bytes: int, G: int, C: int, D: int, block: int, dtype: int,
                         eps: float, stream=None) -> None:
    """Raw C-ABI call: tensors are HOST pointers / CPU tensors, workspace is device memory."""
    _check(lib().la_chunked_step_host(_p(q), _p(k), _p(v), _p(S0), _p(z0), _p(dO), _p(dS_out), _p(dz_out),
                                      _p(o), _p(S_out), _p(z_out), _p(dq), _p(dk), _p(dv), _p(dS0), _p(dz0),
                                      _p(workspace), workspace_bytes, G, C, D, block, dtype, eps, _p(stream)))


def la_bwd_max_c(D: int, block: int, dtype: int) -> int:
    return int(lib().la_bwd_max_c(D, block, dtype))


def la_device_status(clear: bool = True) -> int:
    """Synchronise the device; LA_ERR_TIMEOUT (4) if a kernel gave up a bounded wait,
    LA_ERR_DEVICE (5) if one found its shared memory misaligned (and did nothing) or a
    cross-entropy target was outside [0, V)."""
    return int(lib().la_device_status(1 if clear else 0))


def la_selftest_bounded_wait(wait_us: int = 1000) -> int:
    """Status of the bounded-wait self-test: LA_ERR_TIMEOUT (4) is the expected result."""
    return int(lib().la_selftest_bounded_wait(wait_us))


def la_status_string(status: int) -> str:
    return lib().la_status_string(status).decode()


def la_version() -> int:
    return int(lib().la_version())
