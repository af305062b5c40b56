"""Exit gates: River-LLM cosine gate and TIDE router gate (float64).

Test infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _decide(score: np.ndarray, threshold: float) -> np.ndarray:
    """Strict ``score > threshold`` taken in fp32.

    River-LLM (core method; method step 3) exits when the similarity exceeds
    tau and TIDE (module 3, formula 4) when phi_k exceeds theta: both strict.
    The TIDE notes (module 4) state that its kernels accumulate in fp32, so the
    decision is taken on the fp32-rounded score against the fp32 threshold.
    """
    return (score.astype(np.float32) > np.float32(threshold)).astype(np.uint8)


def cosine_similarity(h_prev, h_cur) -> np.ndarray:
    """State-transition similarity of each token (one row per token).

    River-LLM, background "state transition similarity" and method step 3:
    s_t^(l) = h^(l-1)^T h^(l) / (||h^(l-1)|| ||h^(l)||), the cosine between the
    input and the output of the same decoder block. A zero row has no
    direction; it gets s = 0 (never exits).
    """
    a, b = _f64(h_prev), _f64(h_cur)
    dot = np.einsum("td,td->t", a, b)
    na = np.sqrt(np.einsum("td,td->t", a, a))
    nb = np.sqrt(np.einsum("td,td->t", b, b))
    den = na * nb
    return np.where(den > 0.0, dot / np.where(den > 0.0, den, 1.0), 0.0)


def _apply_rule(score: np.ndarray, threshold: float, rule: str):
    mask = _decide(score, threshold)
    flag = int(mask.size > 0 and bool(mask.all()))
    if rule == "per_token":
        return mask, flag
    if rule == "batch_all":
        return np.full_like(mask, flag), flag
    raise ValueError(rule)


def cosine_gate(h_prev, h_cur, tau: float, rule: str = "per_token"):
    """River-LLM exit check after one backbone layer.

    Method step 3 states the rule as min_{b in B} s > tau over the sequences in
    the batch ("batch_all": one flag, every token exits or none does) and, in
    the same step, says that each token decides on its own ("per_token").
    Both readings are offered. Returns (score, mask, flag) where flag is
    1 iff every token's score exceeds tau, i.e. iff min_b s_b > tau.
    """
    s = cosine_similarity(h_prev, h_cur)
    mask, flag = _apply_rule(s, tau, rule)
    return s, mask, flag


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def router_probability(h, w_down, w_up, gamma=None, b_down=None, b_up=None, eps: float = 1e-5) -> np.ndarray:
    """TIDE router MLP at one checkpoint (formula 3; module 4 kernel).

    p = sigmoid( W_up . SiLU( W_down . RMSNorm(h) + b_down ) + b_up ) with
    W_down in R^{b x d} (b = 128 bottleneck), W_up in R^{1 x b},
    SiLU(x) = x*sigmoid(x), RMSNorm(h) = h / sqrt(mean(h^2) + eps) * gamma.
    The system-architecture section counts d*128 + 128 parameters per
    checkpoint, so gamma defaults to 1 and the biases to 0.
    """
    h = _f64(h)
    w_down = _f64(w_down)
    w_up = _f64(w_up).reshape(-1)
    n, d = h.shape
    b = w_down.shape[0]
    if w_down.shape != (b, d) or w_up.shape != (b,):
        raise ValueError("router weights must be W_down[b][d] and W_up[b]")
    g = np.ones(d) if gamma is None else _f64(gamma)
    r = 1.0 / np.sqrt(np.einsum("td,td->t", h, h) / d + eps)
    hn = h * r[:, None] * g[None, :]
    u = hn @ w_down.T
    if b_down is not None:
        u = u + _f64(b_down)[None, :]
    z = (u * _sigmoid(u)) @ w_up
    if b_up is not None:
        z = z + float(np.asarray(b_up, dtype=np.float64).reshape(-1)[0])
    return _sigmoid(z)


def router_gate(h, w_down, w_up, theta: float, rule: str = "per_token", gamma=None,
                b_down=None, b_up=None, eps: float = 1e-5):
    """TIDE exit decision at one checkpoint: phi_k(H[k+1]) > theta (formula 4).

    Module 3 applies it to every token of the batch at once ("batch_all");
    the compaction kernel of module 4 needs the per-token mask ("per_token").
    Returns (p, mask, flag) with flag = 1 iff every p exceeds theta.
    """
    p = router_probability(h, w_down, w_up, gamma, b_down, b_up, eps)
    mask, flag = _apply_rule(p, theta, rule)
    return p, mask, flag


def earliest_exit(probs: Dict[int, np.ndarray], theta: float, n_layers: int, k_min: int = 0) -> np.ndarray:
    """Exit depth of each token under TIDE's earliest-checkpoint rule (formula 4).

    ``probs[k]`` holds phi_k for checkpoint layer k (0-based; H[k+1] is the
    output of layer k). A token exits at the first checkpoint k >= k_min whose
    probability exceeds theta and then has executed k+1 layers; a token that
    never passes runs all ``n_layers``.
    """
    ks = sorted(probs)
    n = len(probs[ks[0]])
    depth = np.full(n, n_layers, dtype=np.int64)
    done = np.zeros(n, dtype=bool)
    for k in ks:
        if k < k_min:
            continue
        hit = (_decide(_f64(probs[k]), theta) == 1) & ~done
        depth[hit] = k + 1
        done |= hit
    return depth


def layer_ops(depths: Sequence[int]) -> int:
    """Layer executions of a batch whose tokens stop at the given depths
    (TIDE Figure 2 accounting: one layer op per token per executed layer)."""
    return int(np.sum(np.asarray(depths, dtype=np.int64)))
