"""Shared helpers of the GPU parity tests: error measure and tolerances.

Errors are max-norm relative: max|x - y| / max|y| over a tensor (an
elementwise relative error is ill-posed near zero).  Tolerances:
  * fp32 paths: 1e-4 on outputs and states;
  * bf16-input prefill (fp32 state and accumulation): 2e-2 on outputs,
    1e-2 on final and checkpoint states;
  * outputs stored as bf16 by an fp32 path (decode / replay with bf16
    projections): 1e-2, the bf16 storage rounding (2^-9 relative) plus the
    fp32 bound;
  * checkpoint positions, page packing and pack/unpack: bit-exact.
"""
import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16_OUT = 2e-2
TOL_BF16_STATE = 1e-2
TOL_BF16_STORED_OUT = 1e-2


def rel(x, y):
    x = x.detach().to("cpu", torch.float64).numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)
    y = y.detach().to("cpu", torch.float64).numpy() if isinstance(y, torch.Tensor) else np.asarray(y, np.float64)
    assert x.shape == y.shape, (x.shape, y.shape)
    if y.size == 0:
        return 0.0
    denom = np.abs(y).max()
    if denom == 0.0:
        return float(np.abs(x).max())
    return float(np.abs(x - y).max() / denom)
