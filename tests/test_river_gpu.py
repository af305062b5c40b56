"""The Exit River on the GPU (through the C ABI) against the oracle: the hidden
state after every exit layer and the K/V each layer writes, with every other
cache slot untouched."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import river
from tests.parity import check_kv_scaled, f64, host
from workloads import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"

H_REL_L2 = 1e-2
H_MAX_ABS = 5e-2   # at RMS 1; grows with the reference's RMS


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def check_h(gpu, ref, what="h"):
    g = f64(gpu)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    mx = np.abs(g - ref).max(initial=0.0)
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    lim = H_MAX_ABS * max(1.0, rms)
    assert mx <= lim and rel <= H_REL_L2, f"{what}: max-abs {mx:.3e} (bound {lim:.3e}), rel-L2 {rel:.3e}"


def _make(tee, cfg, layers, walk="auto"):
    return tee.ExitRiver(layers, d=cfg.d, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                         d_ff=cfg.d_ff, rope_base=cfg.rope_base, eps=cfg.eps, max_pos=cfg.cache_len, attn=walk)


# the attention's two walks of the cache: whole (item, kv head) pairs, one
# persistent consumer group each (chunks of 128 / 64 positions at head_dim 64 /
# 128), and chunks of 256 / 128 positions, one CTA each, with a split merge
WALKS = ["pair", "chunk"]


def _check(cfg, x, k0, v0, out, items, rows=None):
    """Oracle on the given items (with their rows of h), compared with the GPU's
    h_out[items] and with the written slots; all other slots keep k0 / v0."""
    rows = np.asarray(items if rows is None else rows)
    items = np.asarray(items)
    pos = x["pos"].cpu().numpy()[rows]
    seq = x["seq"].cpu().numpy()[rows]
    layers = host(x["layers"])
    kc, vc = f64(k0), f64(v0)
    ref = river.exit_river(f64(x["h"])[rows], layers, pos, seq, kc, vc, cfg.n_q_heads, cfg.n_kv_heads,
                           cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    check_h(out[torch.as_tensor(items, device=out.device).long()], ref)
    written = torch.zeros(x["k_cache"].shape[:4], dtype=torch.bool, device=DEV)
    ps, ss = torch.as_tensor(pos, device=DEV).long(), torch.as_tensor(seq, device=DEV).long()
    for L in layers:
        j = L["cache_layer"]
        check_kv_scaled(x["k_cache"][j, ss, :, ps], kc[j, seq, :, pos], f"K layer {j}")
        check_kv_scaled(x["v_cache"][j, ss, :, ps], vc[j, seq, :, pos], f"V layer {j}")
        written[j, ss, :, ps] = True
    assert torch.equal(x["k_cache"][~written], k0[~written])
    assert torch.equal(x["v_cache"][~written], v0[~written])


def _cfg(**kw):
    return dataclasses.replace(configs.TINY_RIVER, **kw)


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_river(tee, seed, walk):
    cfg = configs.TINY_RIVER
    x = gen.river_inputs(cfg, seed, DEV)
    k0, v0 = x["k_cache"].clone(), x["v_cache"].clone()
    ws = tee.Workspace(DEV)
    out = _make(tee, cfg, x["layers"], walk)(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"], ws=ws)
    torch.cuda.synchronize()
    assert ws.device_error() == (0, 0)
    _check(cfg, x, k0, v0, out, np.arange(cfg.batch))


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("n_q,n_kv,hd", [(8, 8, 64), (8, 4, 64), (16, 2, 64), (4, 2, 128), (8, 1, 128), (2, 1, 128)])
def test_head_layouts(tee, n_q, n_kv, hd, walk):
    cfg = _cfg(n_q_heads=n_q, n_kv_heads=n_kv, head_dim=hd, d=512, d_ff=320, cache_len=600, batch=5)
    x = gen.river_inputs(cfg, n_q + n_kv + hd, DEV)
    k0, v0 = x["k_cache"].clone(), x["v_cache"].clone()
    out = _make(tee, cfg, x["layers"], walk)(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"])
    _check(cfg, x, k0, v0, out, np.arange(cfg.batch))


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("positions", [[0, 1, 2], [63, 64, 65], [127, 128, 129], [255, 256, 257], [511, 512, 1023]])
def test_chunk_boundaries(tee, positions, walk):
    # chunk edges of both walks at head_dim 64 and 128: 64, 128, 256 positions
    for hd in (64, 128):
        cfg = _cfg(head_dim=hd, n_q_heads=512 // hd, n_kv_heads=256 // hd, d=256, cache_len=1024, batch=3,
                   river_layers=(1,))
        x = gen.river_inputs(cfg, hd + positions[0], DEV)
        x["pos"] = torch.tensor(positions, dtype=torch.int32, device=DEV)
        k0, v0 = x["k_cache"].clone(), x["v_cache"].clone()
        out = _make(tee, cfg, x["layers"], walk)(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"])
        _check(cfg, x, k0, v0, out, np.arange(3))


@pytest.mark.parametrize("walk", WALKS)
@pytest.mark.parametrize("n", [1, 7, 64, 100, 128])
def test_item_counts_rows_and_device_count(tee, n, walk):
    cfg = _cfg(batch=n, cache_len=300)
    x = gen.river_inputs(cfg, n, DEV)
    k0, v0 = x["k_cache"].clone(), x["v_cache"].clone()
    rng = np.random.default_rng(n)
    rows = rng.permutation(n).astype(np.int32)
    n_use = max(1, n - 3)
    n_dev = torch.tensor([n_use], dtype=torch.int32, device=DEV)
    out = torch.full((n, cfg.d), 3.0, dtype=torch.bfloat16, device=DEV)
    _make(tee, cfg, x["layers"], walk)(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"],
                                       rows=torch.from_numpy(rows).to(DEV), n_dev=n_dev, out=out)
    _check(cfg, x, k0, v0, out, np.arange(n_use), rows[:n_use])
    assert bool((out[n_use:] == 3.0).all())


@pytest.mark.parametrize("walk", WALKS)
def test_bad_position_is_recorded_and_skipped(tee, walk):
    cfg = configs.TINY_RIVER
    x = gen.river_inputs(cfg, 5, DEV)
    x["pos"][4] = cfg.cache_len
    k0, v0 = x["k_cache"].clone(), x["v_cache"].clone()
    out = torch.full((cfg.batch, cfg.d), 3.0, dtype=torch.bfloat16, device=DEV)
    ws = tee.Workspace(DEV)
    _make(tee, cfg, x["layers"], walk)(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"], out=out, ws=ws)
    assert ws.device_error() == (2, cfg.cache_len)
    good = np.array([i for i in range(cfg.batch) if i != 4])
    _check(cfg, x, k0, v0, out, good)
    assert bool((out[4] == 3.0).all())


@pytest.mark.parametrize("walk", WALKS)
def test_empty_call_is_a_no_op(tee, walk):
    cfg = configs.TINY_RIVER
    x = gen.river_inputs(cfg, 6, DEV)
    k0 = x["k_cache"].clone()
    n_dev = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((cfg.batch, cfg.d), 3.0, dtype=torch.bfloat16, device=DEV)
    _make(tee, cfg, x["layers"], walk)(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"], n_dev=n_dev,
                                       out=out)
    torch.cuda.synchronize()
    assert torch.equal(x["k_cache"], k0) and bool((out == 3.0).all())


@pytest.mark.parametrize("walk", WALKS)
def test_twice_reuses_the_workspace(tee, walk):
    cfg = configs.TINY_RIVER
    ws = tee.Workspace(DEV)
    for seed in (7, 8):
        x = gen.river_inputs(cfg, seed, DEV)
        k0, v0 = x["k_cache"].clone(), x["v_cache"].clone()
        out = _make(tee, cfg, x["layers"], walk)(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"], ws=ws)
        _check(cfg, x, k0, v0, out, np.arange(cfg.batch))
    assert ws.device_error() == (0, 0)


@pytest.mark.parametrize("walk", ["auto", "chunk"])
def test_llama1b_river_sampled_items(tee, walk):
    # the full workload (64 items, 8 exit layers, 4096 positions) in the launch
    # configuration the benchmark times ("auto": the pair walk, 512 pairs), and on
    # the chunk walk; the oracle runs 3 sampled items, whose sequences it reads
    # (the items' sequences are distinct, so they do not interact)
    cfg = configs.LLAMA1B_RIVER
    x = gen.river_inputs(cfg, 0, DEV)
    f = _make(tee, cfg, x["layers"], walk)
    ws = tee.Workspace(DEV)
    items = np.array([0, 31, 63])
    pos = x["pos"].cpu().numpy()
    P = int(pos[items].max()) + 1
    js = list(cfg.river_layers)
    # the oracle's view: the sampled sequences' first P positions of the exit layers
    it = torch.as_tensor(items, device=DEV)
    k0 = x["k_cache"][js[0]:js[-1] + 1].index_select(1, it)[:, :, :, :P].clone()
    v0 = x["v_cache"][js[0]:js[-1] + 1].index_select(1, it)[:, :, :, :P].clone()
    out = f(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"], ws=ws)
    torch.cuda.synchronize()
    assert ws.device_error() == (0, 0)
    layers = host(x["layers"])
    for i, L in enumerate(layers):
        L["cache_layer"] = i
    kc, vc = f64(k0), f64(v0)
    ref = river.exit_river(f64(x["h"])[items], layers, pos[items], np.arange(3), kc, vc, cfg.n_q_heads,
                           cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    check_h(out[torch.as_tensor(items, device=DEV)], ref, "h_out (sampled)")
    for i, j in enumerate(js):
        for b, it in enumerate(items):
            check_kv_scaled(x["k_cache"][j, it, :, pos[it]], kc[i, b, :, pos[it]], f"K layer {j} item {it}")
            check_kv_scaled(x["v_cache"][j, it, :, pos[it]], vc[i, b, :, pos[it]], f"V layer {j} item {it}")
