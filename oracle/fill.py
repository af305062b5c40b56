"""KV fill for the layers an exiting token skips.

RidgeFill (idea source section): from the split-layer state, a per-layer map
predicts the input of every later layer, and that layer's own projections
write the cache as usual; the map is the closed-form ridge regression of the
"closed-form ridge regression" note, x_j = h_split W_j (no bias). With
W_j = I this is River-LLM's "State Propagation" (motivation section) and
RidgeFill's "identity fill" (measured-results section). River-LLM (method
step 1) keeps the exit layer's KV addressing identical to the backbone, and
stores Wk/Wv as 4-bit weights with fp16 activations (W4A16, background "PTQ").

Argument marshalling over the C++ oracle (``tee_oracle.cpp``), which computes
every value; the only work here is placing the computed rows into the cache
slots they address. Test infrastructure: see the package docstring for who
may import it.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from ._native import f64, i64, lib, ptr, u8


def dequant_int4(packed, scale, zero, group: int = 64) -> np.ndarray:
    """W[k][n] = (q[k][n] - zero[k // group][n]) * scale[k // group][n]: unsigned
    4-bit codes, two per byte along k with even k in the low nibble, fp16 scale
    and fp16 zero per group of ``group`` input rows (the reading of the W4A16
    format River-LLM names)."""
    p = u8(packed)
    half, n = p.shape
    k = 2 * half
    s, z = f64(scale), f64(zero)
    if s.shape != (k // group, n) or z.shape != s.shape or k % group:
        raise ValueError("scale / zero must be [k / group][n]")
    w = np.empty((k, n))
    lib().oc_dequant_int4(k, n, int(group), ptr(p), ptr(s), ptr(z), ptr(w))
    return w


def rms_norm(x, gamma, eps: float) -> np.ndarray:
    """RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma over the last axis."""
    a = f64(x)
    d = a.shape[-1]
    g = f64(np.broadcast_to(f64(gamma), (d,)))
    flat = np.ascontiguousarray(a.reshape(-1, d))
    y = np.empty_like(flat)
    lib().oc_rms_norm(flat.shape[0], d, ptr(flat), ptr(g), float(eps), ptr(y))
    return y.reshape(a.shape)


def rope_rotate_half(k, pos, base: float) -> np.ndarray:
    """Rotary position embedding on the last axis (one head of width hd):
    element i pairs with i + hd/2 and turns by pos * base^(-2i/hd) (positions
    from 0, no frequency scaling, float64). ``pos`` broadcasts against
    k[..., 0]."""
    a = f64(k)
    hd = a.shape[-1]
    p = f64(pos)
    lead = np.broadcast_shapes(a.shape[:-1], p.shape)
    a = np.ascontiguousarray(np.broadcast_to(a, lead + (hd,)).reshape(-1, hd))
    pp = np.ascontiguousarray(np.broadcast_to(p, lead).reshape(-1))
    y = np.empty_like(a)
    lib().oc_rope_rotate_half(a.shape[0], hd, ptr(a), ptr(pp), float(base), ptr(y))
    return y.reshape(lead + (hd,))


def layer_weights(layer: Dict, group: int = 64):
    """Dense float64 (Wk, Wv) of one filled layer, dequantising int4 codes."""
    if layer.get("k_scale") is not None:
        return (dequant_int4(layer["wk"], layer["k_scale"], layer["k_zero"], group),
                dequant_int4(layer["wv"], layer["v_scale"], layer["v_zero"], group))
    return f64(layer["wk"]), f64(layer["wv"])


def fill_rows(h_rows, layer: Dict, pos, n_kv_heads: int, head_dim: int, rope_base: float,
              eps: float, group: int = 64):
    """K and V that filled layer j writes for the given split-layer rows:
    x_j = h W_j (identity when ``w_map`` is None); x^ = RMSNorm_j(x_j);
    k = x^ Wk_j (+ k_bias), v = x^ Wv_j (+ v_bias); with ``k_norm`` each head of
    k is RMS-normalised over head_dim and scaled by k_norm; then RoPE on k at
    each row's position. Returns K, V [rows][n_kv_heads][head_dim] float64."""
    h = f64(h_rows)
    t, d = h.shape
    kvw = n_kv_heads * head_dim
    wm = None if layer.get("w_map") is None else f64(layer["w_map"])
    if wm is not None and wm.shape != (d, d):
        raise ValueError("w_map must be [d][d]")
    g = f64(layer["gamma"]).reshape(d)
    wk, wv = layer_weights(layer, group)
    if wk.shape != (d, kvw) or wv.shape != (d, kvw):
        raise ValueError("Wk / Wv must be [d][n_kv_heads * head_dim]")
    kb = None if layer.get("k_bias") is None else f64(layer["k_bias"]).reshape(kvw)
    vb = None if layer.get("v_bias") is None else f64(layer["v_bias"]).reshape(kvw)
    kn = None if layer.get("k_norm") is None else f64(layer["k_norm"]).reshape(head_dim)
    p = f64(np.broadcast_to(f64(pos).reshape(-1), (t,)))
    k = np.empty((t, n_kv_heads, head_dim))
    v = np.empty((t, n_kv_heads, head_dim))
    lib().oc_fill_rows(t, d, n_kv_heads, head_dim, ptr(h), ptr(wm), ptr(g), ptr(wk), ptr(wv), ptr(kb), ptr(vb),
                       ptr(kn), ptr(p), float(rope_base), float(eps), ptr(k), ptr(v))
    return k, v


def kv_fill(h_split, layers: Sequence[Dict], k_cache, v_cache, n_kv_heads: int, head_dim: int,
            rope_base: float, eps: float, rows: Optional[Sequence[int]] = None,
            pos: Optional[Sequence[int]] = None, pos0: int = 0,
            seq: Optional[Sequence[int]] = None, group: int = 64):
    """Fill every listed layer for every listed split-layer row: item i takes
    row r = rows[i] (or i), position pos[r] (or pos0 + r) and sequence seq[r]
    (or 0), and writes cache[layer.cache_layer][s][head][p][:] in both caches
    ([layers][seqs][kv_heads][positions][head_dim]); every other slot keeps
    its value. A layer with ``writes`` = "k" (or 1) fills only K, "v" (or 2)
    only V. Returns float64 copies of the two caches."""
    h = f64(h_split)
    kc = np.array(f64(k_cache), copy=True)
    vc = np.array(f64(v_cache), copy=True)
    n = h.shape[0] if rows is None else len(rows)
    rr = np.arange(n) if rows is None else i64(rows)
    pp = (pos0 + rr) if pos is None else i64(pos)[rr]
    ss = np.zeros(n, dtype=np.int64) if seq is None else i64(seq)[rr]
    for layer in layers:
        k, v = fill_rows(h[rr], layer, pp, n_kv_heads, head_dim, rope_base, eps, group)
        j = int(layer["cache_layer"])
        w = layer.get("writes")
        for i in range(n):
            if w in (None, 0, "kv", 1, "k"):
                kc[j, ss[i], :, pp[i], :] = k[i]
            if w in (None, 0, "kv", 2, "v"):
                vc[j, ss[i], :, pp[i], :] = v[i]
    return kc, vc
