"""The Exit River: the W4A16 copies of the remaining decoder layers that an
exited token runs through (float64).

River-LLM (core method; method step 1): from the exit layer on, each token
that left the backbone continues through a 4-bit weight copy of every
remaining layer -- its attention and its FFN -- with fp16 activations and an
fp16 KV cache whose addressing (position, head split, dimension layout) is the
backbone's own, so that the pass writes the skipped layers' K/V into the slots
the backbone would have written, and hands its last hidden state to the LM
head. The pages give the layer's parts by name only; the readings taken (a
Llama-style pre-norm block, the decoder the pages measure on):

  x  = RMSNorm(h) * attn_norm
  q, k, v = x Wq, x Wk, x Wv                (W4A16: (q - z) * s per group)
  q, k  <- rotate-half RoPE at the token's position (as the fill)
  cache[layer][seq][kv head][pos] <- k, v   (every item of the call first)
  o_h = softmax(q_h K^T / sqrt(hd)) V       over positions 0..pos of the
                                            token's sequence, q head h reading
                                            kv head h // (n_q / n_kv)
  h1 = h + concat_h(o_h) Wo
  x2 = RMSNorm(h1) * ffn_norm
  h' = h1 + (SiLU(x2 Wg) * (x2 Wu)) Wd      SiLU(a) = a / (1 + e^-a)

Test infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

from typing import Dict, Sequence

import numpy as np

from .fill import dequant_int4, rms_norm, rope_rotate_half

# weight matrices of one exit layer: name -> (codes key, scale key, zero key)
MATS = {m: (f"w{m}", f"{m}_scale", f"{m}_zero") for m in ("q", "k", "v", "o", "g", "u", "d")}


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def weight(layer: Dict, m: str, group: int) -> np.ndarray:
    """Dense float64 weight ``m`` (one of q k v o g u d) of an exit layer,
    [in][out], dequantised from its int4 codes (or taken as given if dense)."""
    w, s, z = MATS[m]
    if layer.get(s) is None:
        return _f64(layer[w])
    return dequant_int4(layer[w], layer[s], layer[z], group)


def silu(a) -> np.ndarray:
    """SiLU(a) = a * sigmoid(a) = a / (1 + exp(-a))."""
    a = _f64(a)
    return a / (1.0 + np.exp(-a))


def attention(q, k_layer, v_layer, pos, seq, n_kv_heads: int) -> np.ndarray:
    """Causal decode attention of each item over its own sequence's cache.

    q [n][n_q][hd]; k_layer, v_layer [n_seq][n_kv][P][hd] (one cache layer);
    item i reads positions 0..pos[i] of sequence seq[i]. Returns o [n][n_q][hd].
    """
    q = _f64(q)
    n, n_q, hd = q.shape
    rep = n_q // n_kv_heads
    o = np.zeros_like(q)
    for i in range(n):
        p, s = int(pos[i]), int(seq[i])
        for h in range(n_q):
            g = h // rep
            kk = _f64(k_layer[s, g, :p + 1])           # [p+1][hd]
            vv = _f64(v_layer[s, g, :p + 1])
            z = kk @ q[i, h] / np.sqrt(hd)
            w = np.exp(z - z.max())
            o[i, h] = (w / w.sum()) @ vv
    return o


def exit_layer(h, layer: Dict, pos, seq, k_cache, v_cache, n_q_heads: int, n_kv_heads: int, head_dim: int,
               rope_base: float, eps: float, group: int = 64) -> np.ndarray:
    """One exit layer over the items h [n][d]. Writes every item's K and V into
    the float64 caches k_cache, v_cache [layers][n_seq][n_kv][P][hd] at
    (layer["cache_layer"], seq, head, pos), then attends; returns h' [n][d]."""
    h = _f64(h)
    n, d = h.shape
    pos = np.asarray(pos, dtype=np.int64)
    seq = np.asarray(seq, dtype=np.int64)
    j = int(layer["cache_layer"])
    x = rms_norm(h, layer["attn_norm"], eps)
    q = (x @ weight(layer, "q", group)).reshape(n, n_q_heads, head_dim)
    k = (x @ weight(layer, "k", group)).reshape(n, n_kv_heads, head_dim)
    v = (x @ weight(layer, "v", group)).reshape(n, n_kv_heads, head_dim)
    q = rope_rotate_half(q, pos[:, None], rope_base)
    k = rope_rotate_half(k, pos[:, None], rope_base)
    for i in range(n):
        k_cache[j, seq[i], :, pos[i]] = k[i]
        v_cache[j, seq[i], :, pos[i]] = v[i]
    o = attention(q, k_cache[j], v_cache[j], pos, seq, n_kv_heads).reshape(n, n_q_heads * head_dim)
    h1 = h + o @ weight(layer, "o", group)
    x2 = rms_norm(h1, layer["ffn_norm"], eps)
    a = silu(x2 @ weight(layer, "g", group)) * (x2 @ weight(layer, "u", group))
    return h1 + a @ weight(layer, "d", group)


def exit_river(h, layers: Sequence[Dict], pos, seq, k_cache, v_cache, n_q_heads: int, n_kv_heads: int,
               head_dim: int, rope_base: float, eps: float, group: int = 64) -> np.ndarray:
    """The items' pass through the exit layers in order: each layer's output is
    the next one's input; returns the last hidden state (for the LM head)."""
    for L in layers:
        h = exit_layer(h, L, pos, seq, k_cache, v_cache, n_q_heads, n_kv_heads, head_dim, rope_base, eps, group)
    return h
