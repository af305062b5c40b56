"""The one-launch small dense KV fill against the oracle, and the generic
CUDA-core kernels (forced with ``generic=True``) on the same calls.

Shapes span the small path's limits: d from 96 to 2048 (one to eight 32-column
passes per CTA of the map), head_dim 32 to 256, fewer heads than CTAs in the
cluster, n_max * d at its 16,384 cap, fp32 / bf16 / fp16, ridge and identity
maps, scrambled gather order, a device item count, and more layers than one
launch takes."""
import numpy as np
import pytest
import torch

from tests.parity import check_decode_fill, check_kv_scaled
from workloads import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def _cfg(dtype, d, hd, n_kv, n, fmap, layers):
    return configs.DecodeConfig(
        name="small-fill", d=d, n_layers=layers, n_q_heads=2 * n_kv, n_kv_heads=n_kv, head_dim=hd, batch=n,
        cache_len=128, gate_layer=0, fill_layers=tuple(range(layers)), tau=0.95, rule="per_token",
        weights="dense", map=fmap, rope_base=1.0e4, dtype=dtype)


def _fill(tee, cfg, x, generic):
    return tee.KVFill(x["layers"], d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                      rope_base=cfg.rope_base, eps=cfg.eps, dtype=x["h_cur"].dtype, max_pos=cfg.cache_len,
                      generic=generic)


SHAPES = [
    # dtype, d, hd, n_kv, n, map, layers
    ("f32", 256, 64, 2, 8, "ridge", 2),       # the tiny decode's shape
    ("f32", 256, 64, 2, 1, "ridge", 1),
    ("bf16", 512, 128, 4, 32, "ridge", 2),    # n_max * d = 16384
    ("bf16", 2048, 64, 8, 8, "identity", 3),  # eight 32-column passes per CTA of the map
    ("f16", 1024, 64, 4, 16, "ridge", 2),
    ("f32", 96, 32, 3, 5, "ridge", 1),        # 12 map columns per CTA, 6 heads for 8 CTAs
    ("bf16", 256, 256, 2, 4, "identity", 2),  # head_dim 256: eight passes per head
    ("f32", 128, 64, 1, 3, "ridge", 70),      # two launches (64 layers each at most)
]


@pytest.mark.parametrize("generic", [False, True], ids=["small", "generic"])
@pytest.mark.parametrize("dtype,d,hd,n_kv,n,fmap,layers", SHAPES)
def test_small_fill_shapes(tee, generic, dtype, d, hd, n_kv, n, fmap, layers):
    cfg = _cfg(dtype, d, hd, n_kv, n, fmap, layers)
    x = gen.decode_inputs(cfg, seed=d + n + layers, device=DEV)
    f = _fill(tee, cfg, x, generic)
    rows = np.random.default_rng(n + hd).permutation(n).astype(np.int32)
    ws = tee.Workspace(DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"],
      ws=ws)
    assert ws.device_error() == (0, 0)
    check_decode_fill(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL)


@pytest.mark.parametrize("generic", [False, True], ids=["small", "generic"])
def test_small_fill_device_count(tee, generic):
    cfg = _cfg("f32", 256, 64, 2, 8, "ridge", 2)
    x = gen.decode_inputs(cfg, seed=3, device=DEV)
    f = _fill(tee, cfg, x, generic)
    rows = np.array([6, 1, 4, 0, 7], dtype=np.int32)
    n_dev = torch.tensor([3], dtype=torch.int32, device=DEV)   # only the first three items
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"],
      n_dev=n_dev, n_max=len(rows))
    check_decode_fill(cfg, x, rows[:3], x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL)


@pytest.mark.parametrize("generic", [False, True], ids=["small", "generic"])
def test_small_fill_bad_position_is_recorded(tee, generic):
    cfg = _cfg("f32", 256, 64, 2, 8, "ridge", 2)
    x = gen.decode_inputs(cfg, seed=4, device=DEV)
    f = _fill(tee, cfg, x, generic)
    pos = x["pos"].clone()
    pos[2] = cfg.cache_len   # one past the last slot
    ws = tee.Workspace(DEV)
    rows = torch.arange(cfg.batch, dtype=torch.int32, device=DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=rows, pos=pos, seq=x["seq"], ws=ws)
    code, detail = ws.device_error()
    assert code == 2 and detail == cfg.cache_len
    good = np.array([r for r in range(cfg.batch) if r != 2], dtype=np.int32)
    check_decode_fill(cfg, x, good, pos.cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL)


@pytest.mark.parametrize("generic", [False, True], ids=["small", "generic"])
def test_small_fill_variants_one_launch(tee, generic):
    """Bias, per-head K norm and a K-only / V-only layer on the small path."""
    cfg = _cfg("bf16", 512, 64, 4, 12, "ridge", 3)
    x = gen.decode_inputs(cfg, seed=9, device=DEV)
    kvw, hd, dt = cfg.kvw, cfg.head_dim, x["h_cur"].dtype
    L0, L1, L2 = x["layers"]
    L0["k_bias"] = gen.normal((kvw,), 0.5, 9, "kb0", DEV, dt)
    L0["v_bias"] = gen.normal((kvw,), 0.5, 9, "vb0", DEV, dt)
    L1["k_norm"] = gen.normal((hd,), 0.2, 9, "kn1", DEV, dt, mean=1.0)
    L1["writes"] = "k"
    L2["writes"] = "v"
    f = _fill(tee, cfg, x, generic)
    rows = np.arange(cfg.batch, dtype=np.int32)[::-1].copy()
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"])
    check_decode_fill(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL,
                      kv_check=check_kv_scaled)
