"""Input activations of the gated delta rule, stated in fp64 NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring).  These are what the
kernels apply in place when asked to take raw inputs ("Flash Linear Attention"
page, sec. 10: the KDA inference backend takes raw tensors and fuses the gate,
the L2 norm of q and k, and sigmoid(beta) into its kernels):

* gate ("KDA source walkthrough", kda_gate_chunk_cumsum, the per-head A_log,
  the optional dt_bias and the optional lower bound):
  without a lower bound  g = -exp(A_log[h]) * softplus(x + dt_bias);
  with lower bound lb    g = lb * sigmoid(exp(A_log[h]) * (x + dt_bias)).
* beta = sigmoid(logit).
* L2 norm per (token, head) over the key dimension, x / max(||x||_2, eps) with
  eps = 1e-12 (the same reading as the workloads' normalisation of q and k).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def softplus(z):
    """log(1 + e^z), evaluated without overflow."""
    z = _f64(z)
    return np.logaddexp(0.0, z)


def sigmoid(z):
    z = _f64(z)
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def gate(x, A_log, dt_bias=None, lower_bound=None):
    """Log-decay from the raw gate input x [B, T, HV] (scalar gate) or [B, T, HV, K] (per channel).

    A_log [HV]; dt_bias [HV] (scalar gate) or [HV, K] (per channel), or None."""
    x = _f64(x)
    A = np.exp(_f64(A_log))
    z = x if dt_bias is None else x + _f64(dt_bias)
    if x.ndim == 3:
        Ab = A[None, None, :]
    else:
        Ab = A[None, None, :, None]
    if lower_bound is None:
        return -Ab * softplus(z)
    return float(lower_bound) * sigmoid(Ab * z)


def beta_from_logits(b):
    return sigmoid(b)


def l2norm(x, eps=1e-12):
    """x / max(||x||_2, eps) over the last axis."""
    x = _f64(x)
    n = np.sqrt((x * x).sum(axis=-1, keepdims=True))
    return x / np.maximum(n, eps)
