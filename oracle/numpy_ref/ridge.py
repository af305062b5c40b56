"""Closed-form ridge fit of a RidgeFill map (float64).

Test infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg


def ridge_fit(X, Y, lam: float) -> np.ndarray:
    """W = (X^T X + lambda I)^-1 X^T Y.

    RidgeFill, "closed-form ridge regression" note: X holds split-layer states,
    Y the true inputs of a later layer, both from one calibration forward pass;
    the map is fitted once in closed form. Solved by a Cholesky factorisation
    of the symmetric positive definite X^T X + lambda I.
    """
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    A = X.T @ X + lam * np.eye(X.shape[1])
    c = scipy.linalg.cho_factor(A, lower=True)
    return scipy.linalg.cho_solve(c, X.T @ Y)
