"""Batch compaction and exit scatter (TIDE, core module 4).

Argument marshalling over the C++ oracle (``tee_oracle.cpp``). Test
infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from ._native import f64, i64, lib, ptr, u8


def stable_partition(mask, pos_in: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """TIDE module 4 "Batch Compact": rows in batch order, exiting (mask != 0)
    to one list, continuing to the other (a stable split); ``pos_in[r]`` (else
    r) is carried into cont_pos / exit_pos for the later scatter."""
    m = u8(np.asarray(mask) != 0)
    n = m.shape[0]
    pin = None if pos_in is None else i64(pos_in).reshape(n)
    out = {k: np.empty(n, dtype=np.int64) for k in ("cont_rows", "exit_rows", "cont_pos", "exit_pos")}
    counts = np.empty(2, dtype=np.int64)
    lib().oc_stable_partition(n, ptr(m), ptr(pin), ptr(out["cont_rows"]), ptr(out["exit_rows"]),
                              ptr(out["cont_pos"]), ptr(out["exit_pos"]), ptr(counts))
    nc, ne = int(counts[0]), int(counts[1])
    return {"cont_rows": out["cont_rows"][:nc], "exit_rows": out["exit_rows"][:ne],
            "cont_pos": out["cont_pos"][:nc], "exit_pos": out["exit_pos"][:ne], "counts": counts}


def gather_rows(h, rows) -> np.ndarray:
    """The compacted buffer of continuing tokens: row i is h[rows[i]] (float64)."""
    a = f64(h)
    r = i64(rows).reshape(-1)
    if r.size and (r.min() < 0 or r.max() >= a.shape[0]):
        raise IndexError("row out of range")
    out = np.empty((r.shape[0], a.shape[1]))
    lib().oc_gather_rows(r.shape[0], a.shape[1], ptr(a), ptr(r), ptr(out))
    return out


def exit_scatter(out, h_src, exit_rows, exit_pos, gamma=None, eps: float = 1e-5) -> np.ndarray:
    """Exit scatter (TIDE module 4): out[exit_pos[i]] = h_src[exit_rows[i]]; with
    ``gamma`` the row first goes through the final RMSNorm ("Exit Projection").
    Returns a float64 copy of ``out`` with the rows replaced."""
    res = np.array(f64(out), copy=True)
    src = f64(h_src)
    er, ep = i64(exit_rows).reshape(-1), i64(exit_pos).reshape(-1)
    g = None if gamma is None else f64(gamma).reshape(src.shape[1])
    if er.shape != ep.shape or res.ndim != 2 or res.shape[1] != src.shape[1]:
        raise ValueError("exit_rows / exit_pos / out do not match")
    if er.size and (er.min() < 0 or er.max() >= src.shape[0] or ep.min() < 0 or ep.max() >= res.shape[0]):
        raise IndexError("row or slot out of range")
    lib().oc_exit_scatter(er.shape[0], src.shape[1], ptr(src), ptr(er), ptr(ep), ptr(g), float(eps), ptr(res))
    return res
