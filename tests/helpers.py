"""Shared helpers of the GPU parity tests: tolerance checks against the oracle."""
import numpy as np
import torch

# Tolerances stated for the path: max|gpu - ref| / max|ref| <= 1e-5 for float32
# inputs, <= 2e-3 for bfloat16 inputs with the float32 state.  A bfloat16
# OUTPUT additionally carries its own rounding (unit roundoff 2^-8), so
# bfloat16 outputs are checked element-wise against 2e-3 max|ref| + 2^-8 |ref|.
TOL_F32 = 1e-5
TOL_BF16 = 2e-3


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(gpu, ref):
    gpu, ref = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    scale = max(float(np.max(np.abs(ref))) if ref.size else 0.0, 1e-30)
    return float(np.max(np.abs(gpu - ref))) / scale if ref.size else 0.0


def assert_close(gpu, ref, in_dtype, out_dtype=None, what=""):
    """Assert the stated bound for this input/output precision."""
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    out_dtype = out_dtype or torch.float32
    tol = TOL_F32 if in_dtype == torch.float32 else TOL_BF16
    if out_dtype == torch.bfloat16:
        scale = np.max(np.abs(r)) if r.size else 0.0
        bound = tol * scale + 2.0 ** -8 * np.abs(r)
        bad = np.abs(g - r) > bound
        assert not bad.any(), f"{what}: {bad.sum()} elements beyond bound, worst excess " \
                              f"{np.max(np.abs(g - r) - bound):.3e}"
    else:
        e = rel_err(g, r)
        assert e <= tol, f"{what}: rel err {e:.3e} > {tol:.1e}"
