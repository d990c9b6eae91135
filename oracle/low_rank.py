"""Float64 CPU oracle for the low-rank projection (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this module; the product path (the CUDA library and its Python binding) never does.

What it computes (module neuralops.core.triton_kernels.low_rank, functions ``fwd`` and
``bwd``): with x [M, K_in], V [r, K_in], U [K_out, r] and an optional bias [K_out],

    t = x V^T            [M, r]       (the low-rank bottleneck)
    y = t U^T + bias     [M, K_out]

and the gradient of ``fwd`` (the page's ``bwd`` differentiates ``fwd`` with autograd) for an
output gradient g [M, K_out]:

    dt = g U,  dx = dt V,  dU = g^T t,  dV = dt^T x,  dbias = sum over the rows of g.

The definition is written out as it stands, in float64, with numpy matrix products as the
steps (no blocking, fusion or reordering).  Leading dimensions of x (batch, sequence) are
flattened into the M rows, as the projection treats every row alike.

Parity: pinned by tests/test_oracle_low_rank.py (explicit index sums on tiny inputs, the
identity-weight and rank-one special cases, the merged-weight contraction order, central
finite differences of the forward, homogeneity identities of the gradients).
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def _check(x, U, V, bias):
    if x.ndim < 1 or U.ndim != 2 or V.ndim != 2:
        raise ValueError("x [..., K_in], U [K_out, r], V [r, K_in]")
    r, k_in = V.shape
    k_out, r2 = U.shape
    if x.shape[-1] != k_in or r2 != r:
        raise ValueError(f"shapes disagree: x {x.shape}, U {U.shape}, V {V.shape}")
    if bias is not None and bias.shape != (k_out,):
        raise ValueError("bias must have K_out elements")


def fwd(x, U, V, bias=None) -> np.ndarray:
    """y = (x V^T) U^T + bias, float64, with x's leading dimensions kept."""
    x, U, V, bias = (_f64(a) for a in (x, U, V, bias))
    _check(x, U, V, bias)
    lead = x.shape[:-1]
    xm = x.reshape(-1, x.shape[-1])
    t = xm @ V.T
    y = t @ U.T
    if bias is not None:
        y = y + bias[None, :]
    return y.reshape(lead + (U.shape[0],))


def bwd(x, U, V, grad_out, bias=None):
    """(dx, dU, dV, dbias) of y = (x V^T) U^T + bias for the output gradient grad_out;
    dbias is None without a bias."""
    x, U, V, g, bias = (_f64(a) for a in (x, U, V, grad_out, bias))
    _check(x, U, V, bias)
    lead = x.shape[:-1]
    xm = x.reshape(-1, x.shape[-1])
    gm = g.reshape(-1, U.shape[0])
    t = xm @ V.T
    dt = gm @ U
    dx = dt @ V
    dU = gm.T @ t
    dV = dt.T @ xm
    db = gm.sum(axis=0) if bias is not None else None
    return dx.reshape(lead + (x.shape[-1],)), dU, dV, db
