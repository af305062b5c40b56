"""Closed-form ridge fit of a RidgeFill map.

Argument marshalling over the C++ oracle (``tee_oracle.cpp``). Test
infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

import numpy as np

from ._native import f64, lib, ptr


def ridge_fit(X, Y, lam: float) -> np.ndarray:
    """W = (X^T X + lambda I)^-1 X^T Y (RidgeFill, "closed-form ridge
    regression" note: X the split-layer states, Y a later layer's true inputs,
    from one calibration pass), by a Cholesky factorisation of X^T X + lambda I
    and two triangular solves. Raises numpy.linalg.LinAlgError when that
    matrix is not positive definite."""
    x, y = f64(X), f64(Y)
    if y.ndim == 1:
        y = y[:, None]
    y = np.ascontiguousarray(y)
    n, d = x.shape
    if y.shape[0] != n:
        raise ValueError("X and Y need the same rows")
    w = np.empty((d, y.shape[1]))
    if lib().oc_ridge_fit(n, d, y.shape[1], ptr(x), ptr(y), float(lam), ptr(w)) != 0:
        raise np.linalg.LinAlgError("X^T X + lambda I is not positive definite")
    return w if np.asarray(Y).ndim == 2 else w[:, 0]
