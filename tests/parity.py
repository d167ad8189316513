"""Shared helpers of the GPU parity tests: tolerance check and host <-> device conversions."""

import numpy as np
import torch

MAX_ABS = 2e-2    # bf16 outputs, fp32 accumulation
MEAN_ABS = 2e-3


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def assert_close(gpu, ref, what, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    d = np.abs(g - r)
    mx, mn = float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3e} (<= {max_abs}), mean-abs {mn:.3e} (<= {mean_abs})"
    return mx, mn
