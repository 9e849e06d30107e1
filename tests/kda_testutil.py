"""Helpers shared by the GPU parity tests (comparison metric, sampling)."""
import numpy as np
import torch

# Tolerances on max|x - x_ref| / rms(x_ref), per output tensor.
TOL_BF16 = 2e-3   # bf16 inputs, fp32 state and fp32 output
TOL_F32 = 1e-5    # fp32 inputs


def rel_err(x, ref) -> float:
    """max |x - ref| / rms(ref), in fp64; NaN anywhere gives inf."""
    x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if not np.all(np.isfinite(x)):
        return float("inf")
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(x - ref))) / max(rms, 1e-300)


def tol_for(dtype) -> float:
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def to_dev(d: dict, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
