"""Comparison helpers shared by the parity tests.

Metric (the reading used for "max relative error"): per tensor,
    max_i |x_i - ref_i| / max_i |ref_i|
(normwise max-relative).  Elementwise relative error is ill-posed here because v
has zero mean, so outputs pass through zero.
"""
import numpy as np

# Tolerances: float32 inputs 1e-4 on every output; bfloat16 inputs with float32
# accumulation 2e-2 on o, dq, dk, dv and 1e-2 on the carry and its gradients.
TOL = {
    "f32": {"o": 1e-4, "S_out": 1e-4, "z_out": 1e-4, "dq": 1e-4, "dk": 1e-4, "dv": 1e-4, "dS0": 1e-4, "dz0": 1e-4},
    "bf16": {"o": 2e-2, "S_out": 1e-2, "z_out": 1e-2, "dq": 2e-2, "dk": 2e-2, "dv": 2e-2, "dS0": 1e-2, "dz0": 1e-2},
}


def to_np(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def max_rel(x, ref):
    x, ref = to_np(x), to_np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    scale = np.abs(ref).max()
    assert np.isfinite(x).all(), "non-finite values in the CUDA result"
    return float(np.abs(x - ref).max() / max(scale, 1e-30))


def check(results, refs, dtype, names):
    errs = {n: max_rel(r, f) for n, r, f in zip(names, results, refs)}
    bad = {n: (e, TOL[dtype][n]) for n, e in errs.items() if not e <= TOL[dtype][n]}
    assert not bad, f"parity failed (error, tolerance): {bad}; all: {errs}"
    return errs
