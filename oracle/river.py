"""The Exit River: the W4A16 copies of the remaining decoder layers that an
exited token runs through.

River-LLM (core method; method step 1): from the exit layer on, each token
that left the backbone continues through a 4-bit weight copy of every
remaining layer -- its attention and its FFN -- with fp16 activations and a KV
cache whose addressing is the backbone's own, so that the pass writes the
skipped layers' K/V into the slots the backbone would have written. The pages
name the layer's parts only; the block is read as the Llama pre-norm block of
the decoder they measure on:

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

Argument marshalling over the C++ oracle (``tee_oracle.cpp``). Test
infrastructure: see the package docstring for who may import it.
"""
from __future__ import annotations

from typing import Dict, Sequence

import numpy as np

from ._native import f64, i64, lib, ptr
from .fill import dequant_int4

# weight matrices of one exit layer: name -> (codes key, scale key, zero key)
MATS = {m: (f"w{m}", f"{m}_scale", f"{m}_zero") for m in ("q", "k", "v", "o", "g", "u", "d")}


def weight(layer: Dict, m: str, group: int) -> np.ndarray:
    """Dense float64 weight ``m`` (one of q k v o g u d) of an exit layer,
    [in][out], dequantised from its int4 codes (or taken as given if dense)."""
    w, s, z = MATS[m]
    if layer.get(s) is None:
        return f64(layer[w])
    return dequant_int4(layer[w], layer[s], layer[z], group)


def silu(a) -> np.ndarray:
    """SiLU(a) = a * sigmoid(a) = a / (1 + exp(-a)), elementwise."""
    x = f64(a)
    flat = np.ascontiguousarray(x.reshape(-1))
    y = np.empty_like(flat)
    lib().oc_silu(flat.shape[0], ptr(flat), ptr(y))
    return y.reshape(x.shape)


def attention(q, k_layer, v_layer, pos, seq, n_kv_heads: int) -> np.ndarray:
    """Causal decode attention of each item over its own sequence's cache:
    q [n][n_q][hd]; k_layer, v_layer [n_seq][n_kv][P][hd]; item i reads
    positions 0..pos[i] of sequence seq[i]. Returns o [n][n_q][hd]."""
    qq = f64(q)
    kl, vl = f64(k_layer), f64(v_layer)
    n, n_q, hd = qq.shape
    n_seq, n_kv, P, hd2 = kl.shape
    p, s = i64(pos).reshape(n), i64(seq).reshape(n)
    if n_kv != n_kv_heads or hd2 != hd or vl.shape != kl.shape or n_q % n_kv:
        raise ValueError("head layout mismatch")
    if n and (p.min() < 0 or p.max() >= P or s.min() < 0 or s.max() >= n_seq):
        raise IndexError("position or sequence out of range")
    o = np.empty_like(qq)
    lib().oc_attention(n, n_q, hd, ptr(qq), ptr(kl), ptr(vl), n_kv, P, ptr(p), ptr(s), ptr(o))
    return o


def exit_layer(h, layer: Dict, pos, seq, k_cache, v_cache, n_q_heads: int, n_kv_heads: int, head_dim: int,
               rope_base: float, eps: float, group: int = 64) -> np.ndarray:
    """One exit layer over the items h [n][d]. Writes every item's K and V into
    the float64 caches k_cache, v_cache [layers][n_seq][n_kv][P][hd] (numpy,
    updated in place) at (layer["cache_layer"], seq, head, pos), then attends;
    returns h' [n][d]."""
    hh = f64(h)
    n, d = hh.shape
    j = int(layer["cache_layer"])
    p, s = i64(pos).reshape(n), i64(seq).reshape(n)
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.dtype == np.float64 and c.flags.c_contiguous):
            raise TypeError("the caches must be C-contiguous float64 numpy arrays (updated in place)")
    _, n_seq, n_kv, P, hd = k_cache.shape
    if (n_kv, hd) != (n_kv_heads, head_dim) or v_cache.shape != k_cache.shape:
        raise ValueError("cache layout mismatch")
    if n and (p.min() < 0 or p.max() >= P or s.min() < 0 or s.max() >= n_seq):
        raise IndexError("position or sequence out of range")
    kl, vl = k_cache[j], v_cache[j]   # contiguous views: written in place
    W = {m: weight(layer, m, group) for m in MATS}
    d_ff = W["g"].shape[1]
    an, fn = f64(layer["attn_norm"]).reshape(d), f64(layer["ffn_norm"]).reshape(d)
    out = np.empty_like(hh)
    lib().oc_exit_layer(n, d, n_q_heads, n_kv_heads, head_dim, d_ff, ptr(hh), ptr(an), ptr(fn), ptr(W["q"]),
                        ptr(W["k"]), ptr(W["v"]), ptr(W["o"]), ptr(W["g"]), ptr(W["u"]), ptr(W["d"]), ptr(p),
                        ptr(s), P, ptr(kl), ptr(vl), float(rope_base), float(eps), ptr(out))
    return out


def exit_river(h, layers: Sequence[Dict], pos, seq, k_cache, v_cache, n_q_heads: int, n_kv_heads: int,
               head_dim: int, rope_base: float, eps: float, group: int = 64) -> np.ndarray:
    """The items' pass through the exit layers in order: each layer's output is
    the next one's input; returns the last hidden state (for the LM head)."""
    for L in layers:
        h = exit_layer(h, L, pos, seq, k_cache, v_cache, n_q_heads, n_kv_heads, head_dim, rope_base, eps, group)
    return h
