"""KV fill for the layers an exiting token skips (float64).

RidgeFill (idea source section): from the split-layer state, a per-layer map
predicts the input of every later layer, and that layer's own projections
write the cache as usual. The map is the closed-form ridge regression of the
"closed-form ridge regression" note, x_j = h_split W_j (no bias). With
W_j = I this is River-LLM's "State Propagation" (motivation section) and
RidgeFill's "identity fill" (measured-results section). River-LLM (method
step 1) keeps the exit layer's KV addressing (position index, head split,
dimension layout) identical to the backbone, and stores Wk/Wv as 4-bit
weights with fp16 activations (W4A16, background "PTQ").

Test infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def dequant_int4(packed, scale, zero, group: int = 64) -> np.ndarray:
    """W[k][n] = (q[k][n] - zero[k // group][n]) * scale[k // group][n].

    River-LLM's exit layers hold 4-bit weights with fp16 activations (W4A16,
    background "PTQ"; method step 1 names HQQ without giving its format). The
    reading used: unsigned codes 0..15, two per byte along the input dimension
    k with even k in the low nibble, fp16 scale and fp16 (fractional) zero per
    group of ``group`` consecutive input rows.
    """
    p = np.asarray(packed, dtype=np.uint8)
    half, kvw = p.shape
    q = np.empty((2 * half, kvw), dtype=np.float64)
    q[0::2] = (p & 0x0F).astype(np.float64)
    q[1::2] = (p >> 4).astype(np.float64)
    s = np.repeat(_f64(scale), group, axis=0)
    z = np.repeat(_f64(zero), group, axis=0)
    return (q - z) * s


def rms_norm(x, gamma, eps: float) -> np.ndarray:
    """RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma, row by row."""
    x = _f64(x)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * r * _f64(gamma)


def rope_rotate_half(k, pos, base: float) -> np.ndarray:
    """Rotary position embedding on the last axis (one head of width hd).

    The pages name no convention (River-LLM only requires the exit layer to
    write what the backbone would). The reading used is the "rotate-half"
    pairing of element i with i + hd/2, angle pos * base^(-2i/hd), positions
    counted from 0, no frequency scaling, all in float64.
    ``k`` has shape [..., hd]; ``pos`` broadcasts against k[..., 0].
    """
    k = _f64(k)
    hd = k.shape[-1]
    half = hd // 2
    inv_freq = base ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = _f64(pos)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = k[..., :half], k[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def layer_weights(layer: Dict, group: int = 64):
    """Dense float64 (Wk, Wv) of one filled layer, dequantising int4 codes."""
    if layer.get("k_scale") is not None:
        wk = dequant_int4(layer["wk"], layer["k_scale"], layer["k_zero"], group)
        wv = dequant_int4(layer["wv"], layer["v_scale"], layer["v_zero"], group)
        return wk, wv
    return _f64(layer["wk"]), _f64(layer["wv"])


def fill_rows(h_rows, layer: Dict, pos, n_kv_heads: int, head_dim: int, rope_base: float,
              eps: float, group: int = 64):
    """K and V that filled layer j writes for the given split-layer rows.

    x_j = h W_j (identity when ``w_map`` is None); x^ = RMSNorm_j(x_j);
    k = x^ Wk_j (+ k_bias), v = x^ Wv_j (+ v_bias); with ``k_norm`` every head of
    k is RMS-normalised over head_dim (same eps) and scaled by k_norm; then k
    gets RoPE at each row's position, per kv head. The bias and the K norm are
    the QKV-bias and QK-norm model families that RidgeFill's notes cover.
    Returns K, V of shape [rows][n_kv_heads][head_dim] in float64.
    """
    h = _f64(h_rows)
    x = h if layer.get("w_map") is None else h @ _f64(layer["w_map"])
    xn = rms_norm(x, layer["gamma"], eps)
    wk, wv = layer_weights(layer, group)
    t = h.shape[0]
    k = xn @ wk
    v = xn @ wv
    if layer.get("k_bias") is not None:
        k = k + _f64(layer["k_bias"])
    if layer.get("v_bias") is not None:
        v = v + _f64(layer["v_bias"])
    k = k.reshape(t, n_kv_heads, head_dim)
    v = v.reshape(t, n_kv_heads, head_dim)
    if layer.get("k_norm") is not None:
        k = rms_norm(k, layer["k_norm"], eps)
    k = rope_rotate_half(k, np.asarray(pos, dtype=np.float64)[:, None], rope_base)
    return k, v


def kv_fill(h_split, layers: Sequence[Dict], k_cache, v_cache, n_kv_heads: int, head_dim: int,
            rope_base: float, eps: float, rows: Optional[Sequence[int]] = None,
            pos: Optional[Sequence[int]] = None, pos0: int = 0,
            seq: Optional[Sequence[int]] = None, group: int = 64):
    """Fill every listed layer for every listed split-layer row.

    Item i takes row r = rows[i] (or i) of ``h_split``, position
    p = pos[r] (or pos0 + r) and sequence s = seq[r] (or 0), and writes
    cache[layer.cache_layer][s][head][p][:] for every kv head, in both caches.
    Caches are [layers][seqs][kv_heads][positions][head_dim]; every other slot
    keeps its value. A layer with ``writes`` = "k" (or 1) fills only the K cache,
    "v" (or 2) only the V cache. Returns float64 copies of the two caches.
    """
    h = _f64(h_split)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    n = h.shape[0] if rows is None else len(rows)
    rr = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    pp = (pos0 + rr) if pos is None else np.asarray(pos, dtype=np.int64)[rr]
    ss = np.zeros(n, dtype=np.int64) if seq is None else np.asarray(seq, dtype=np.int64)[rr]
    for layer in layers:
        k, v = fill_rows(h[rr], layer, pp, n_kv_heads, head_dim, rope_base, eps, group)
        L = int(layer["cache_layer"])
        w = layer.get("writes")
        write_k = w in (None, 0, "kv", 1, "k")
        write_v = w in (None, 0, "kv", 2, "v")
        for i in range(n):
            if write_k:
                kc[L, ss[i], :, pp[i], :] = k[i]
            if write_v:
                vc[L, ss[i], :, pp[i], :] = v[i]
    return kc, vc
