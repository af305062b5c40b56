"""Model-family variants of the KV fill on the GPU against the oracle: K and V
bias (QKV-bias models), a per-head RMSNorm of K before RoPE (QK-norm models),
and layers that fill only the K or only the V cache. Each of the three fill
paths is covered: the generic kernels (fp32), the tcgen05 prefill (dense bf16)
and the tcgen05 decode (int4 W4A16).

K and V here are checked with ``check_kv_scaled``: a K bias or a per-head K
norm lifts the reference's RMS from about 0.5 to about 1, and the fill's
roundings are relative errors, so the max-abs bound scales with that RMS
(relative L2 stays 1e-2)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import check_decode_fill, check_kv_scaled, f64, host
from workloads import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (k_bias, v_bias, k_norm, writes) per layer, cycled over the filled layers
VARIANTS = {
    "qkv_bias": [(True, True, False, None)],
    "qk_norm": [(False, False, True, None)],
    "bias_and_norm": [(True, True, True, None)],
    "k_only_v_only": [(False, False, True, "k"), (False, True, False, "v")],
    "v_only_first": [(False, True, False, "v"), (True, False, True, None)],
}


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def _add_variants(layers, kvw, hd, dtype, seed, kind):
    spec = VARIANTS[kind]
    for i, L in enumerate(layers):
        kb, vb, kn, w = spec[i % len(spec)]
        if kb:
            L["k_bias"] = gen.normal((kvw,), 0.5, seed, f"kb{i}", DEV, dtype)
        if vb:
            L["v_bias"] = gen.normal((kvw,), 0.5, seed, f"vb{i}", DEV, dtype)
        if kn:
            L["k_norm"] = gen.normal((hd,), 0.2, seed, f"kn{i}", DEV, dtype, mean=1.0)
        if w:
            L["writes"] = w
    return layers


def _make(tee, cfg, layers, dtype, max_pos, int4=False, generic=False):
    return tee.KVFill(layers, d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, rope_base=cfg.rope_base,
                      eps=cfg.eps, dtype=dtype, max_pos=max_pos, int4=int4, group=getattr(cfg, "group", 64),
                      generic=generic)


@pytest.mark.parametrize("kind", sorted(VARIANTS))
def test_generic_fill_variants(tee, kind):
    cfg = configs.TINY_DECODE
    x = gen.decode_inputs(cfg, seed=11, device=DEV)
    _add_variants(x["layers"], cfg.n_kv_heads * cfg.head_dim, cfg.head_dim, torch.float32, 11, kind)
    f = _make(tee, cfg, x["layers"], torch.float32, cfg.cache_len, generic=True)
    rows = np.array([5, 0, 7, 2, 3], dtype=np.int32)
    ws = tee.Workspace(DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"], ws=ws)
    assert ws.device_error() == (0, 0)
    check_decode_fill(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL,
                      kv_check=check_kv_scaled)


@pytest.mark.parametrize("kind", sorted(VARIANTS))
@pytest.mark.parametrize("n,hd,d", [(64, 64, 2048), (48, 128, 2048), (7, 128, 1024), (100, 64, 512)])
def test_decode_int4_fill_variants(tee, kind, n, hd, d):
    base = configs.LLAMA1B_DECODE
    cfg = configs.DecodeConfig(**{**base.__dict__, "d": d, "batch": n, "head_dim": hd, "n_kv_heads": 512 // hd,
                                  "n_layers": 4, "fill_layers": (1, 2, 3)})
    x = gen.decode_inputs(cfg, seed=n + hd, device=DEV, case="exit")
    _add_variants(x["layers"], cfg.n_kv_heads * hd, hd, torch.bfloat16, n, kind)
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.cache_len, int4=True)
    rows = np.random.default_rng(n).permutation(n).astype(np.int32)
    ws = tee.Workspace(DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"], ws=ws)
    assert ws.device_error() == (0, 0)
    check_decode_fill(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL,
                      kv_check=check_kv_scaled)


def test_decode_v_only_first_layer_still_records_bad_positions(tee):
    # the clusters of the K half of layer 0 leave at once: another CTA reports
    cfg = configs.LLAMA1B_DECODE
    x = gen.decode_inputs(cfg, seed=4, device=DEV, case="exit")
    _add_variants(x["layers"], cfg.n_kv_heads * cfg.head_dim, cfg.head_dim, torch.bfloat16, 4, "v_only_first")
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.cache_len, int4=True)
    pos = x["pos"].clone()
    pos[9] = cfg.cache_len
    rows = torch.arange(cfg.batch, dtype=torch.int32, device=DEV)
    ws = tee.Workspace(DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=rows, pos=pos, seq=x["seq"], ws=ws)
    assert ws.device_error() == (2, cfg.cache_len)
    good = np.array([r for r in range(cfg.batch) if r != 9], dtype=np.int32)
    check_decode_fill(cfg, x, good, pos.cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL,
                      kv_check=check_kv_scaled)


def _tc_layers(cfg, n_layers, seed, identity):
    import math
    d, kvw = cfg.d, cfg.kvw
    out = []
    for i in range(n_layers):
        w = None if identity else (gen.normal((d, d), 1.0 / math.sqrt(d), seed, f"W{i}", DEV) +
                                   0.5 * torch.eye(d, device=DEV)).bfloat16()
        out.append({"cache_layer": i, "w_map": w,
                    "gamma": gen.normal((d,), 0.1, seed, f"g{i}", DEV, torch.bfloat16, mean=1.0),
                    "wk": gen.normal((d, kvw), math.sqrt(0.25 / d), seed, f"wk{i}", DEV, torch.bfloat16),
                    "wv": gen.normal((d, kvw), math.sqrt(0.25 / d), seed, f"wv{i}", DEV, torch.bfloat16)})
    return out


@pytest.mark.parametrize("kind", sorted(VARIANTS))
@pytest.mark.parametrize("hd,identity", [(128, False), (64, True)])
def test_tc_prefill_fill_variants(tee, kind, hd, identity):
    cfg = configs.PrefillFillConfig(name="variants", d=1024, n_layers=2, n_q_heads=16, n_kv_heads=512 // hd,
                                    head_dim=hd, rope_base=1e6, split=0, tokens=1024, exact_tail=0)
    rows, pos0 = 600, 37
    h = gen.normal((rows, cfg.d), 1.0, 5, "h", DEV, torch.bfloat16)
    layers = _add_variants(_tc_layers(cfg, 2, 5, identity), cfg.kvw, hd, torch.bfloat16, 5, kind)
    shape = (2, 1, cfg.n_kv_heads, cfg.tokens, hd)
    kc = torch.full(shape, gen.CACHE_SENTINEL, dtype=torch.bfloat16, device=DEV)
    vc = kc.clone()
    f = _make(tee, cfg, layers, torch.bfloat16, cfg.tokens)
    ws = tee.Workspace(DEV)
    f(h, kc, vc, pos0=pos0, ws=ws)
    assert ws.device_error() == (0, 0)
    check = np.unique(np.concatenate([np.arange(32), np.arange(rows - 32, rows),
                                      np.random.default_rng(hd).integers(0, rows, 64)])).astype(np.int64)
    hh = f64(h[torch.as_tensor(check, device=DEV)])
    p = torch.as_tensor(pos0 + check, device=DEV)
    for L, Lh in zip(layers, host(layers)):
        k_ref, v_ref = oracle.fill_rows(hh, Lh, pos0 + check, cfg.n_kv_heads, hd, cfg.rope_base, cfg.eps)
        j = L["cache_layer"]
        for c, cache, ref in (("k", kc, k_ref), ("v", vc, v_ref)):
            got = cache[j, 0].index_select(1, p).permute(1, 0, 2)
            if L.get("writes") in (None, c):
                check_kv_scaled(got, ref, f"{c.upper()} layer {j}")
            else:   # the other cache keeps what the backbone wrote
                assert bool((cache[j] == gen.CACHE_SENTINEL).all())
    for cache in (kc, vc):
        assert bool((cache[:, :, :, :pos0] == gen.CACHE_SENTINEL).all())
        assert bool((cache[:, :, :, pos0 + rows:] == gen.CACHE_SENTINEL).all())
