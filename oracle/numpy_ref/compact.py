"""Batch compaction and exit scatter (TIDE, core module 4).

Test infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from .fill import rms_norm


def stable_partition(mask, pos_in: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Split the rows of a batch into continuing and exiting tokens.

    TIDE core module 4 ("Batch Compact") separates continuing from exiting
    tokens. Written as the plain loop over rows in order, so both lists keep
    the batch order (a stable split). ``pos_in[r]`` is the original slot of
    local row r (identity when absent); it is carried into cont_pos/exit_pos
    so that a later scatter finds the original output rows.
    """
    mask = np.asarray(mask)
    n = mask.shape[0]
    pos = np.arange(n, dtype=np.int64) if pos_in is None else np.asarray(pos_in, dtype=np.int64)
    cont, exit_ = [], []
    for r in range(n):
        if mask[r] != 0:
            exit_.append(r)
        else:
            cont.append(r)
    cont_rows = np.array(cont, dtype=np.int64)
    exit_rows = np.array(exit_, dtype=np.int64)
    return {"cont_rows": cont_rows, "exit_rows": exit_rows,
            "cont_pos": pos[cont_rows] if cont else np.zeros(0, np.int64),
            "exit_pos": pos[exit_rows] if exit_ else np.zeros(0, np.int64),
            "counts": np.array([len(cont), len(exit_)], dtype=np.int64)}


def gather_rows(h, rows) -> np.ndarray:
    """The compacted buffer of continuing tokens: row i is h[rows[i]]."""
    h = np.asarray(h)
    return np.stack([h[r] for r in rows]) if len(rows) else h[:0].copy()


def exit_scatter(out, h_src, exit_rows, exit_pos, gamma=None, eps: float = 1e-5) -> np.ndarray:
    """Exit scatter (TIDE module 4): out[exit_pos[i]] = h_src[exit_rows[i]].

    Rows of ``out`` that no exiting token targets keep their values. With
    ``gamma`` the copied row first goes through the final RMSNorm, which is
    the "Exit Projection" kernel of the same module (RMSNorm fused with the
    scatter). Returns a float64 copy of ``out`` with the rows replaced.
    """
    res = np.array(out, dtype=np.float64, copy=True)
    src = np.asarray(h_src, dtype=np.float64)
    for i in range(len(exit_rows)):
        row = src[exit_rows[i]]
        if gamma is not None:
            row = rms_norm(row[None, :], gamma, eps)[0]
        res[exit_pos[i]] = row
    return res
