"""Seeded synthetic inputs for the five workloads.

Both sides of every parity check draw their inputs here: the CUDA library gets
the tensors on the device, the oracle gets the same values widened to float64
on the host. This module only draws random numbers, casts them to the storage
dtype and packs int4 codes two to a byte; it holds none of the method's
arithmetic (no cosine, no norm, no projection, no rotation).

Every tensor comes from its own ``torch.Generator`` whose seed is a stable
hash of (seed, tensor tag), so that a tensor does not change when another one
is added or resized. The values depend on the device the generator runs on
(CPU and CUDA use different streams); a test draws all its inputs on one
device and copies them across when both sides need them.

Distributions (the pages give none; these are the readings used):
  * hidden states ~ N(0, 1); decode pairs h_cur = a*h_prev + sqrt(1-a^2)*N(0, 1)
    with a ~ Beta(8, 1) drawn as u**(1/8), u ~ U(0, 1);
  * ridge maps W_j ~ N(0, 1/d) (tiny decode) or N(0, 1/d) + 0.5*I (prefill);
  * layer-norm weights g_j = 1 + 0.1*N(0, 1);
  * dense Wk, Wv ~ N(0, 0.25/d), so that |K|, |V| stay well below 4;
  * int4 Wk, Wv: codes q ~ U{0..15}, fp16 zero z = 7.5 + U(-0.5, 0.5) and fp16
    scale s = sqrt(0.25/d)/sqrt(21.25) * (1 + 0.1*N(0, 1)) per group of 64
    input rows, which gives the dequantised weights about the dense spread;
  * router weights ~ N(0, 0.02^2), gamma = 1, no biases;
  * Exit River layers: every weight int4 as above (spread sqrt(0.25/d_in)),
    norm weights 1 + 0.1*N(0, 1); cache history K, V ~ N(0, 0.5^2).
"""
from __future__ import annotations

import math
import zlib
from typing import Dict, List, Optional

import torch

from .configs import DecodeConfig, PrefillFillConfig, RiverConfig, RouterConfig

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}

# Sentinel written into every cache slot before a fill, so that a test can
# tell written slots from untouched ones. Exactly representable in bf16/f32.
CACHE_SENTINEL = -7.0


def _rng(seed: int, tag: str, device) -> torch.Generator:
    key = zlib.crc32(f"{seed}:{tag}".encode()) ^ (seed * 0x9E3779B1 & 0xFFFFFFFF)
    g = torch.Generator(device=device)
    g.manual_seed(int(key))
    return g


def normal(shape, std, seed, tag, device, dtype=torch.float32, mean=0.0):
    g = _rng(seed, tag, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(dtype)


def uniform(shape, lo, hi, seed, tag, device):
    g = _rng(seed, tag, device)
    u = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
    return u.mul_(hi - lo).add_(lo)


def randint(shape, lo, hi, seed, tag, device, dtype=torch.int32):
    g = _rng(seed, tag, device)
    return torch.randint(lo, hi, shape, generator=g, device=device, dtype=torch.int64).to(dtype)


def pack_int4(q: torch.Tensor) -> torch.Tensor:
    """Pack codes q[k][n] in 0..15 two per byte along k: even k in the low nibble."""
    assert q.shape[0] % 2 == 0
    lo = q[0::2].to(torch.uint8)
    hi = q[1::2].to(torch.uint8)
    return lo | (hi << 4)


def int4_weight(d: int, kvw: int, group: int, seed: int, tag: str, device) -> Dict[str, torch.Tensor]:
    q = randint((d, kvw), 0, 16, seed, tag + ".q", device, dtype=torch.uint8)
    s0 = math.sqrt(0.25 / d) / math.sqrt(21.25)
    scale = normal((d // group, kvw), 0.1 * s0, seed, tag + ".s", device, mean=s0).to(torch.float16)
    zero = uniform((d // group, kvw), 7.0, 8.0, seed, tag + ".z", device).to(torch.float16)
    return {"packed": pack_int4(q), "scale": scale, "zero": zero}


def _beta8_1(n, seed, tag, device):
    return uniform((n,), 0.0, 1.0, seed, tag, device).pow_(1.0 / 8.0)


def decode_inputs(cfg: DecodeConfig, seed: int = 0, device="cpu", case: str = "default",
                  with_cache: bool = True) -> Dict[str, object]:
    """Inputs of one decode step.

    ``case`` (bf16 batch-min workload only): "exit" draws a ~ U(0.985, 1) for
    every token, so that the batch-min rule fires; "stay" is the same with
    token 0 at a = 0.5, so that it does not. "default" draws a ~ Beta(8, 1).
    """
    n, d, kvw, dt = cfg.batch, cfg.d, cfg.kvw, _DT[cfg.dtype]
    h_prev = normal((n, d), 1.0, seed, "h_prev", device)
    noise = normal((n, d), 1.0, seed, "h_noise", device)
    if case == "default":
        a = _beta8_1(n, seed, "a", device)
    else:
        a = uniform((n,), 0.985, 1.0, seed, "a", device)
        if case == "stay":
            a[0] = 0.5
        elif case != "exit":
            raise ValueError(case)
    h_cur = a[:, None] * h_prev + torch.sqrt(1.0 - a * a)[:, None] * noise
    pos = randint((n,), 0, cfg.cache_len, seed, "pos", device)
    layers: List[Dict[str, Optional[torch.Tensor]]] = []
    for j in cfg.fill_layers:
        L: Dict[str, Optional[torch.Tensor]] = {"cache_layer": j}
        L["w_map"] = (None if cfg.map == "identity"
                      else normal((d, d), 1.0 / math.sqrt(d), seed, f"W{j}", device, dt))
        L["gamma"] = normal((d,), 0.1, seed, f"g{j}", device, dt, mean=1.0)
        if cfg.weights == "dense":
            L["wk"] = normal((d, kvw), math.sqrt(0.25 / d), seed, f"wk{j}", device, dt)
            L["wv"] = normal((d, kvw), math.sqrt(0.25 / d), seed, f"wv{j}", device, dt)
        else:
            k = int4_weight(d, kvw, cfg.group, seed, f"wk{j}", device)
            v = int4_weight(d, kvw, cfg.group, seed, f"wv{j}", device)
            L.update(wk=k["packed"], wv=v["packed"], k_scale=k["scale"], k_zero=k["zero"],
                     v_scale=v["scale"], v_zero=v["zero"])
        layers.append(L)
    out = {"h_prev": h_prev.to(dt), "h_cur": h_cur.to(dt), "a": a, "pos": pos,
           "seq": torch.arange(n, dtype=torch.int32, device=device), "layers": layers}
    if with_cache:
        shape = (cfg.n_layers, n, cfg.n_kv_heads, cfg.cache_len, cfg.head_dim)
        out["k_cache"] = torch.full(shape, CACHE_SENTINEL, dtype=dt, device=device)
        out["v_cache"] = torch.full(shape, CACHE_SENTINEL, dtype=dt, device=device)
    return out


def router_weights(cfg: RouterConfig, checkpoint: int, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    dt, b, d = _DT[cfg.dtype], cfg.bottleneck, cfg.d
    return {"w_down": normal((b, d), cfg.weight_std, seed, f"wd{checkpoint}", device, dt),
            "w_up": normal((b,), cfg.weight_std, seed, f"wu{checkpoint}", device, dt)}


def router_hidden(cfg: RouterConfig, n: int, checkpoint: int, seed: int = 0, device="cpu") -> torch.Tensor:
    return normal((n, cfg.d), 1.0, seed, f"h{checkpoint}:{n}", device, _DT[cfg.dtype])


def prefill_inputs(cfg: PrefillFillConfig, seed: int = 0, device="cpu", rows: Optional[int] = None,
                   layers: Optional[int] = None, with_cache: bool = True) -> Dict[str, object]:
    """Inputs of a RidgeFill prefill fill. ``rows``/``layers`` shrink the
    workload (same distributions) for tests that do not need the full size."""
    d, kvw, dt = cfg.d, cfg.kvw, _DT[cfg.dtype]
    n = cfg.filled_rows if rows is None else rows
    fill = cfg.fill_layers if layers is None else cfg.fill_layers[:layers]
    h = normal((n, d), 1.0, seed, f"h_split:{n}", device, dt)
    eye = torch.eye(d, device=device, dtype=torch.float32)
    Ls = []
    for i, j in enumerate(fill):
        w = normal((d, d), 1.0 / math.sqrt(d), seed, f"W{j}", device)
        w.add_(eye, alpha=0.5)
        Ls.append({"cache_layer": i, "w_map": w.to(dt),
                   "gamma": normal((d,), 0.1, seed, f"g{j}", device, dt, mean=1.0),
                   "wk": normal((d, kvw), math.sqrt(0.25 / d), seed, f"wk{j}", device, dt),
                   "wv": normal((d, kvw), math.sqrt(0.25 / d), seed, f"wv{j}", device, dt)})
        del w
    del eye
    out = {"h_split": h, "layers": Ls}
    if with_cache:
        shape = (len(fill), 1, cfg.n_kv_heads, cfg.tokens, cfg.head_dim)
        out["k_cache"] = torch.full(shape, CACHE_SENTINEL, dtype=dt, device=device)
        out["v_cache"] = torch.full(shape, CACHE_SENTINEL, dtype=dt, device=device)
    return out


def river_positions(cfg: RiverConfig, seed: int = 0, device="cpu") -> torch.Tensor:
    """The exited tokens' cache positions, U[0, cache_len) per sequence."""
    return randint((cfg.batch,), 0, cfg.cache_len, seed, "pos", device)


def river_inputs(cfg: RiverConfig, seed: int = 0, device="cpu", with_cache: bool = True,
                 dtype=torch.bfloat16) -> Dict[str, object]:
    """Inputs of one Exit River pass: the exited tokens' hidden states, their
    positions and sequences, the W4A16 layers, and caches whose history
    (every slot) holds random values that the attention reads."""
    n, d, f = cfg.batch, cfg.d, cfg.d_ff
    h = normal((n, d), 1.0, seed, "h_exit", device, dtype)
    pos = river_positions(cfg, seed, device)
    layers: List[Dict[str, object]] = []
    for j in cfg.river_layers:
        L: Dict[str, object] = {"cache_layer": j}
        L["attn_norm"] = normal((d,), 0.1, seed, f"an{j}", device, dtype, mean=1.0)
        L["ffn_norm"] = normal((d,), 0.1, seed, f"fn{j}", device, dtype, mean=1.0)
        for m, (k_in, n_out) in {"q": (d, cfg.qw), "k": (d, cfg.kvw), "v": (d, cfg.kvw), "o": (cfg.qw, d),
                                 "g": (d, f), "u": (d, f), "d": (f, d)}.items():
            w = int4_weight(k_in, n_out, cfg.group, seed, f"w{m}{j}", device)
            L[f"w{m}"], L[f"{m}_scale"], L[f"{m}_zero"] = w["packed"], w["scale"], w["zero"]
        layers.append(L)
    out = {"h": h, "pos": pos, "seq": torch.arange(n, dtype=torch.int32, device=device), "layers": layers}
    if with_cache:
        shape = (cfg.n_layers, n, cfg.n_kv_heads, cfg.cache_len, cfg.head_dim)
        out["k_cache"] = normal(shape, 0.5, seed, "k_hist", device, dtype)
        out["v_cache"] = normal(shape, 0.5, seed, "v_hist", device, dtype)
    return out


def ridge_inputs(n: int, d: int, seed: int = 0, device="cpu") -> Dict[str, torch.Tensor]:
    """Calibration rows for a ridge map: X ~ N(0, 1) [n][d] and Y = X A + 0.1 N(0, 1)
    with A ~ N(0, 1/d) + 0.5 I (the prefill maps' distribution), both bf16."""
    x = normal((n, d), 1.0, seed, f"ridge_x:{n}x{d}", device)
    a = normal((d, d), 1.0 / math.sqrt(d), seed, f"ridge_a:{d}", device)
    a += 0.5 * torch.eye(d, device=device)
    y = x @ a + normal((n, d), 0.1, seed, f"ridge_e:{n}x{d}", device)
    return {"x": x.to(torch.bfloat16), "y": y.to(torch.bfloat16)}
