"""Shared helpers for the GPU tests: tolerances and tensor <-> numpy glue.

Tolerances (stated once, used by every parity test):
  |delta log pi|           <= 5e-3  (absolute, per token)
  loss, D3                 <= 1e-4  relative (abs floor 1e-7 for values near 0)
  dH, dW                   <= 1e-2  relative L2 (Frobenius) error
"""

import numpy as np
import torch

TOL_LOGPI = 5e-3
TOL_SCALAR_REL = 1e-4
TOL_SCALAR_ABS = 1e-7
TOL_GRAD_REL_L2 = 1e-2


def f64(t):
    """Exact float64 copy of a (bf16/fp32/int) tensor on the host."""
    if t.dtype in (torch.int32, torch.int64):
        return t.detach().cpu().numpy().astype(np.int64)
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def scalar_close(got, want, rel=TOL_SCALAR_REL, abs_floor=TOL_SCALAR_ABS):
    return abs(got - want) <= max(rel * abs(want), abs_floor)


def bits(t):
    """fp32 tensor -> int32 bit patterns on the host (for bitwise checks)."""
    return t.detach().cpu().contiguous().view(torch.int32).numpy()
