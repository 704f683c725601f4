"""Shared pieces of the GPU parity tests: tolerances and device marshalling."""
from __future__ import annotations

import numpy as np
import torch

from oracle_pins import rel_err  # noqa: F401  (the tolerance metric, one definition)

# Tolerances on max_i |g - r| / max(|r_i|, rms(r)) per output tensor.
# fp32 inputs: 1e-4 on y and state. bf16 inputs (the oracle sees the same
# bf16-rounded values): 2e-3 on y, and 1e-4 on the state, where only the
# fp32-versus-fp64 arithmetic differs.
RTOL_F32 = 1e-4
RTOL_Y_BF16 = 2e-3
RTOL_STATE = 1e-4


def y_tol(in_dtype) -> float:
    return RTOL_F32 if in_dtype == torch.float32 else RTOL_Y_BF16


def to_dev(d, device):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()
