"""fp64 gate projection: the gate logits a = x W^T + b from the layer input.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The bounded gate is g = -5 sigmoid(projection(x)) ("Architecture Analysis of Ultra-Long
Context Sparse MoE Models", §2.2; "From Numerical Stability to Load Balancing", §2.2);
the projection is a linear layer, so its definition is one matrix product plus a bias,
written here in fp64 with NumPy's matmul (a library primitive). Inputs are converted to
fp64 first; bf16 values convert exactly.
"""
from __future__ import annotations

import numpy as np


def _f64(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        import torch
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def gate_projection(x, weight, bias=None):
    """``x`` [N, d_model], ``weight`` [n_out, d_model], ``bias`` [n_out] or None ->
    ``a`` [N, n_out] fp64."""
    x, w, b = _f64(x), _f64(weight), _f64(bias)
    a = x @ w.T
    return a if b is None else a + b[None, :]
