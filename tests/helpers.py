"""Shared test helpers: tolerances, conversions, the library fixture logic."""
import numpy as np
import torch

# Tolerances of the parity contract: max|gpu - ref| / max|ref| over the whole
# tensor, for fp32 inputs (CUDA-core path) and for bf16 inputs (fp32 state and
# accumulation, bf16 tensor-core operands).
TOL_F32 = 1e-5
TOL_BF16 = 2e-2


def relmax(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    den = np.max(np.abs(ref)) if ref.size else 1.0
    if den == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / den)


def f64(t):
    """Exact float64 copy of a tensor (bf16 and fp32 widen exactly)."""
    return t.detach().to("cpu", torch.float64).numpy()


def tol_for(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16
