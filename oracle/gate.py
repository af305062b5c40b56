"""Exit gates: River-LLM cosine gate and TIDE router gate.

Argument marshalling over the C++ oracle (``tee_oracle.cpp``): every value is
computed there, in float64 loops. Test infrastructure: see the package
docstring for who may import it.
"""
from __future__ import annotations

from typing import Dict

import numpy as np

from ._native import f64, i64, lib, ptr

_RULES = {"per_token": 0, "batch_all": 1}


def _rows(x) -> np.ndarray:
    a = f64(x)
    if a.ndim != 2:
        raise ValueError("expected [tokens][d]")
    return a


def _apply_rule(score: np.ndarray, threshold: float, rule: str):
    """Strict ``score > threshold`` in fp32 (River-LLM core method "exceeds
    tau"; TIDE formula 4; TIDE module 4's fp32 accumulation); flag = every
    token exits; under the batch rule every mask entry equals the flag."""
    if rule not in _RULES:
        raise ValueError(rule)
    s = f64(score)
    mask = np.empty(s.shape[0], dtype=np.uint8)
    flag = np.zeros(1, dtype=np.int32)
    lib().oc_decide(s.shape[0], ptr(s), float(threshold), _RULES[rule], ptr(mask), ptr(flag))
    return mask, int(flag[0])


def cosine_similarity(h_prev, h_cur) -> np.ndarray:
    """State-transition similarity of each token (River-LLM, background "state
    transition similarity" and method step 3): the cosine between the input
    and the output of the same block; a zero row gets 0."""
    a, b = _rows(h_prev), _rows(h_cur)
    if a.shape != b.shape:
        raise ValueError("h_prev and h_cur differ in shape")
    s = np.empty(a.shape[0])
    lib().oc_cosine_similarity(a.shape[0], a.shape[1], ptr(a), ptr(b), ptr(s))
    return s


def cosine_gate(h_prev, h_cur, tau: float, rule: str = "per_token"):
    """River-LLM exit check after one backbone layer (method step 3): the
    batch rule min_b s > tau ("batch_all") or each token on its own
    ("per_token"). Returns (score, mask, flag), flag = 1 iff min_b s > tau."""
    s = cosine_similarity(h_prev, h_cur)
    mask, flag = _apply_rule(s, tau, rule)
    return s, mask, flag


def router_probability(h, w_down, w_up, gamma=None, b_down=None, b_up=None, eps: float = 1e-5) -> np.ndarray:
    """TIDE router MLP at one checkpoint (formula 3; module 4 "Fused LayerNorm +
    Route"): p = sigmoid(W_up . SiLU(W_down . RMSNorm(h) + b_down) + b_up),
    W_down [b][d], W_up [b]; gamma defaults to 1 and the biases to 0."""
    h = _rows(h)
    wd = f64(w_down)
    wu = f64(w_up).reshape(-1)
    n, d = h.shape
    b = wd.shape[0]
    if wd.shape != (b, d) or wu.shape != (b,):
        raise ValueError("router weights must be W_down[b][d] and W_up[b]")
    g = None if gamma is None else f64(gamma).reshape(d)
    bd = None if b_down is None else f64(b_down).reshape(b)
    bu = None if b_up is None else f64(b_up).reshape(-1)[:1]
    p = np.empty(n)
    lib().oc_router_probability(n, d, b, ptr(h), ptr(wd), ptr(wu), ptr(g), ptr(bd), ptr(bu), float(eps), ptr(p))
    return p


def router_gate(h, w_down, w_up, theta: float, rule: str = "per_token", gamma=None,
                b_down=None, b_up=None, eps: float = 1e-5):
    """TIDE exit decision at one checkpoint, phi_k(H[k+1]) > theta (formula 4);
    module 3 applies it to all tokens at once ("batch_all"), module 4's
    compaction needs it per token. Returns (p, mask, flag)."""
    p = router_probability(h, w_down, w_up, gamma, b_down, b_up, eps)
    mask, flag = _apply_rule(p, theta, rule)
    return p, mask, flag


def earliest_exit(probs: Dict[int, np.ndarray], theta: float, n_layers: int, k_min: int = 0) -> np.ndarray:
    """Exit depth of each token under TIDE's earliest-checkpoint rule (formula
    4): ``probs[k]`` is phi_k at 0-based checkpoint layer k; a token exits at
    the first k >= k_min whose probability exceeds theta, having run k + 1
    layers, else it runs all ``n_layers``."""
    ks = sorted(probs)
    kk = i64(ks)
    P = f64(np.stack([f64(probs[k]).reshape(-1) for k in ks]))
    n = P.shape[1]
    depth = np.empty(n, dtype=np.int64)
    lib().oc_earliest_exit(len(ks), ptr(kk), n, ptr(P), float(theta), int(n_layers), int(k_min), ptr(depth))
    return depth


def layer_ops(depths) -> int:
    """Layer executions of a batch whose tokens stop at the given depths (TIDE
    Figure 2: one layer op per token per executed layer)."""
    d = i64(depths).reshape(-1)
    return int(lib().oc_layer_ops(d.shape[0], ptr(d)))
