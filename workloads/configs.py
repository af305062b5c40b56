"""Shapes and hyper-parameters of the five synthetic workloads.

Each workload stands in for the kind of run the three source pages measure:
decode at small batch (River-LLM: Llama-3.2-1B / Llama-3.1-8B at batch 1 on an
A40), a per-checkpoint router over a prefill batch (TIDE: d=4096 models on an
A100), and long-context prefill KV fill (RidgeFill: 16K-120K tokens). No
dataset, prompt or trained weight is used: every tensor is drawn by
``workloads.gen`` from a seeded generator.

This module holds sizes only; it contains none of the method's arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Tuple


@dataclass(frozen=True)
class DecodeConfig:
    """One decode step: gate -> compaction -> KV fill -> exit scatter."""
    name: str
    d: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    batch: int                 # tokens in the step, one per sequence
    cache_len: int             # positions per sequence in the cache
    gate_layer: int            # 0-based layer whose output is h_cur
    fill_layers: Tuple[int, ...]   # 0-based layers that the exit fills
    tau: float
    rule: str                  # "per_token" or "batch_all"
    weights: str               # "dense" or "int4"
    map: str                   # "ridge" (W_j ~ N(0,1/d)) or "identity"
    rope_base: float
    dtype: str                 # "f32" or "bf16"
    group: int = 64
    eps: float = 1e-5

    @property
    def kvw(self) -> int:
        return self.n_kv_heads * self.head_dim


@dataclass(frozen=True)
class RouterConfig:
    """Router gate + compaction at one checkpoint (TIDE)."""
    name: str
    d: int
    n_layers: int
    checkpoints: Tuple[int, ...]
    bottleneck: int
    thetas: Tuple[float, ...]
    batches: Tuple[int, ...]
    weight_std: float = 0.02
    dtype: str = "bf16"
    eps: float = 1e-5


@dataclass(frozen=True)
class PrefillFillConfig:
    """RidgeFill prefill: fill every layer after the split for the leading rows."""
    name: str
    d: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    rope_base: float
    split: int                 # layers [0, split) run exactly
    tokens: int                # prompt length T
    exact_tail: int            # last rows kept exact (not filled)
    dtype: str = "bf16"
    eps: float = 1e-5

    @property
    def kvw(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def fill_layers(self) -> Tuple[int, ...]:
        return tuple(range(self.split, self.n_layers))

    @property
    def filled_rows(self) -> int:
        return self.tokens - self.exact_tail


@dataclass(frozen=True)
class RiverConfig:
    """The Exit River of one decode step: the exited tokens through the W4A16
    copies of layers river_layers (River-LLM)."""
    name: str
    d: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    batch: int                 # exited tokens, one per sequence
    cache_len: int
    river_layers: Tuple[int, ...]
    rope_base: float
    group: int = 64
    eps: float = 1e-5

    @property
    def kvw(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qw(self) -> int:
        return self.n_q_heads * self.head_dim


# Tiny Exit River: two layers of a d=256 model, 8 tokens, 128 cache positions.
TINY_RIVER = RiverConfig(
    name="tiny-river", d=256, n_layers=4, n_q_heads=4, n_kv_heads=2, head_dim=64, d_ff=512,
    batch=8, cache_len=128, river_layers=(2, 3), rope_base=1.0e4)

# Llama-3.2-1B-shaped Exit River: 64 tokens that exited after layer 8 run the
# W4A16 copies of layers 9-16 (0-based 8-15), 4096 cache positions.
LLAMA1B_RIVER = RiverConfig(
    name="llama3.2-1b-exit-river-w4a16", d=2048, n_layers=16, n_q_heads=32, n_kv_heads=8, head_dim=64,
    d_ff=8192, batch=64, cache_len=4096, river_layers=tuple(range(8, 16)), rope_base=5.0e5)


# Tiny fp32 decode step: exit after 1-based layer 2, fill 1-based layers 3-4.
TINY_DECODE = DecodeConfig(
    name="tiny-fp32-decode", d=256, n_layers=4, n_q_heads=4, n_kv_heads=2,
    head_dim=64, batch=8, cache_len=128, gate_layer=1, fill_layers=(2, 3),
    tau=0.95, rule="per_token", weights="dense", map="ridge",
    rope_base=1.0e4, dtype="f32")

# Llama-3.2-1B-shaped decode, bf16, batch-min cosine gate after layer 8,
# identity map (state propagation) and int4 group-64 Wk/Wv.
LLAMA1B_DECODE = DecodeConfig(
    name="llama3.2-1b-decode-w4a16", d=2048, n_layers=16, n_q_heads=32,
    n_kv_heads=8, head_dim=64, batch=64, cache_len=4096, gate_layer=7,
    fill_layers=tuple(range(8, 16)), tau=0.97, rule="batch_all",
    weights="int4", map="identity", rope_base=5.0e5, dtype="bf16")

# TIDE router at every 4th layer of a 32-layer d=4096 model.
ROUTER_4096 = RouterConfig(
    name="router-d4096", d=4096, n_layers=32,
    checkpoints=tuple(k for k in range(32) if (k + 1) % 4 == 0),
    bottleneck=128, thetas=(0.5, 0.6, 0.7, 0.8, 0.9), batches=(32, 4096))

# RidgeFill 16K prefill on a d=4096 32-layer model.
PREFILL_16K = PrefillFillConfig(
    name="prefill-fill-16k", d=4096, n_layers=32, n_q_heads=32, n_kv_heads=8,
    head_dim=128, rope_base=5.0e5, split=16, tokens=16384, exact_tail=2048)

# RidgeFill 120K prefill on a d=5120 64-layer model.
PREFILL_120K = PrefillFillConfig(
    name="prefill-fill-120k", d=5120, n_layers=64, n_q_heads=40, n_kv_heads=8,
    head_dim=128, rope_base=1.0e6, split=32, tokens=122880, exact_tail=4096)

ALL = {c.name: c for c in (TINY_DECODE, LLAMA1B_DECODE, ROUTER_4096,
                           PREFILL_16K, PREFILL_120K, TINY_RIVER, LLAMA1B_RIVER)}
