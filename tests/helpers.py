"""Shared test helpers: tolerances and comparisons against the oracle."""
import numpy as np
import torch

# Tolerances on max|gpu - oracle| / max|oracle| over a whole tensor: fp32
# inputs 1e-4, bf16 inputs (fp32 state) 2e-2.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_err(got, ref) -> float:
    got = got.detach().to("cpu", torch.float64).numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    denom = np.abs(ref).max()
    assert np.isfinite(got).all(), "non-finite values in the GPU result"
    return float(np.abs(got - ref).max() / max(denom, 1e-30))
