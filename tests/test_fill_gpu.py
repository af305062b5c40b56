"""KV fill on the GPU (through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import check_decode_fill, check_kv, f64, host
from workloads import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def _make(tee, cfg, layers, dtype, max_pos, int4=False):
    return tee.KVFill(layers, d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, rope_base=cfg.rope_base,
                      eps=cfg.eps, dtype=dtype, max_pos=max_pos, int4=int4, group=getattr(cfg, "group", 64))


def _check_decode(cfg, x, rows, pos, seq):
    check_decode_fill(cfg, x, rows, pos, seq, gen.CACHE_SENTINEL)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32_decode_fill(tee, seed):
    cfg = configs.TINY_DECODE
    x = gen.decode_inputs(cfg, seed=seed, device=DEV)
    f = _make(tee, cfg, x["layers"], torch.float32, cfg.cache_len)
    rows = np.array([r for r in range(cfg.batch) if (r + seed) % 3 != 0], dtype=np.int32)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"])
    _check_decode(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy())


@pytest.mark.parametrize("seed", [0, 1])
def test_llama1b_w4a16_identity_fill(tee, seed):
    cfg = configs.LLAMA1B_DECODE
    x = gen.decode_inputs(cfg, seed=seed, device=DEV, case="exit")
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.cache_len, int4=True)
    rows = np.arange(cfg.batch, dtype=np.int32)
    n_dev = torch.tensor([cfg.batch], dtype=torch.int32, device=DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"],
      n_dev=n_dev, n_max=cfg.batch)
    _check_decode(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy())


def test_device_count_limits_the_items(tee):
    cfg = configs.LLAMA1B_DECODE
    x = gen.decode_inputs(cfg, seed=5, device=DEV, case="exit")
    f = _make(tee, cfg, x["layers"][:2], torch.bfloat16, cfg.cache_len, int4=True)
    rows = np.array([63, 5, 17, 40, 2], dtype=np.int32)
    n_dev = torch.tensor([3], dtype=torch.int32, device=DEV)   # only the first three items
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"],
      n_dev=n_dev, n_max=len(rows))
    x["layers"] = x["layers"][:2]
    _check_decode(cfg, x, rows[:3], x["pos"].cpu().numpy(), x["seq"].cpu().numpy())


def _prefill_check(cfg, x, rows_checked, n_rows, pos0=0):
    h = f64(x["h_split"][torch.as_tensor(rows_checked, device=DEV).long()])
    for L, Lh in zip(x["layers"], host(x["layers"])):
        k_ref, v_ref = oracle.fill_rows(h, Lh, pos0 + rows_checked, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base,
                                        cfg.eps)
        j = L["cache_layer"]
        p = torch.as_tensor(pos0 + rows_checked, device=DEV).long()
        # [kv_heads][rows][hd] -> [rows][kv_heads][hd]
        check_kv(x["k_cache"][j, 0].index_select(1, p).permute(1, 0, 2), k_ref, f"K layer {j}")
        check_kv(x["v_cache"][j, 0].index_select(1, p).permute(1, 0, 2), v_ref, f"V layer {j}")
    for c in (x["k_cache"], x["v_cache"]):
        assert bool((c[:, :, :, :pos0] == gen.CACHE_SENTINEL).all())
        assert bool((c[:, :, :, pos0 + n_rows:] == gen.CACHE_SENTINEL).all())


@pytest.mark.parametrize("rows,layers", [(1, 1), (127, 1), (300, 2), (1000, 2)])
def test_prefill_fill_small_cases(tee, rows, layers):
    cfg = configs.PREFILL_16K
    x = gen.prefill_inputs(cfg, seed=rows, device=DEV, rows=rows, layers=layers)
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.tokens)
    f(x["h_split"], x["k_cache"], x["v_cache"])
    check = np.unique(np.concatenate([np.arange(min(rows, 64)), np.arange(max(0, rows - 64), rows),
                                      np.random.default_rng(rows).integers(0, rows, 64)])).astype(np.int64)
    _prefill_check(cfg, x, check, rows)


def test_prefill_fill_with_position_offset(tee):
    cfg = configs.PREFILL_16K
    x = gen.prefill_inputs(cfg, seed=9, device=DEV, rows=200, layers=1)
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.tokens)
    f(x["h_split"], x["k_cache"], x["v_cache"], pos0=1000)
    _prefill_check(cfg, x, np.arange(200), 200, pos0=1000)


def test_bad_positions_are_recorded_and_skipped(tee):
    cfg = configs.TINY_DECODE
    x = gen.decode_inputs(cfg, seed=3, device=DEV)
    ws = tee.Workspace(DEV)
    f = _make(tee, cfg, x["layers"], torch.float32, cfg.cache_len)
    pos = x["pos"].clone()
    pos[2] = cfg.cache_len + 5
    rows = torch.arange(cfg.batch, dtype=torch.int32, device=DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=rows, pos=pos, seq=x["seq"], ws=ws)
    code, detail = ws.device_error()
    assert code == 2 and detail == cfg.cache_len + 5   # TEE_DEVERR_POS
    good = np.array([r for r in range(cfg.batch) if r != 2], dtype=np.int32)
    _check_decode(cfg, x, good, pos.cpu().numpy(), x["seq"].cpu().numpy())


# ---------------------------------------------------------------- tensor-core path
# bf16 fills of at least 256 rows with dense weights run on tcgen05 (128 x 256 tiles).

def _layers_for(cfg, d, kvw, n_layers, seed, identity=False):
    import math
    out = []
    for i in range(n_layers):
        w = None if identity else (gen.normal((d, d), 1.0 / math.sqrt(d), seed, f"W{i}", DEV) +
                                   0.5 * torch.eye(d, device=DEV)).bfloat16()
        out.append({"cache_layer": i, "w_map": w,
                    "gamma": gen.normal((d,), 0.1, seed, f"g{i}", DEV, torch.bfloat16, mean=1.0),
                    "wk": gen.normal((d, kvw), math.sqrt(0.25 / d), seed, f"wk{i}", DEV, torch.bfloat16),
                    "wv": gen.normal((d, kvw), math.sqrt(0.25 / d), seed, f"wv{i}", DEV, torch.bfloat16)})
    return out


@pytest.mark.parametrize("rows", [256, 257, 383, 640, 4109])
def test_tc_fill_ragged_tails(tee, rows):
    cfg = configs.PREFILL_16K
    x = gen.prefill_inputs(cfg, seed=rows, device=DEV, rows=rows, layers=2)
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.tokens)
    f(x["h_split"], x["k_cache"], x["v_cache"])
    rng = np.random.default_rng(rows)
    check = np.unique(np.concatenate([np.arange(40), np.arange(rows - 40, rows), rng.integers(0, rows, 48)]))
    _prefill_check(cfg, x, check.astype(np.int64), rows)


@pytest.mark.parametrize("identity", [True, False])
def test_tc_fill_head_dim_64_and_identity_map(tee, identity):
    cfg = configs.PrefillFillConfig(name="hd64", d=2048, n_layers=4, n_q_heads=32, n_kv_heads=8, head_dim=64,
                                    rope_base=5e5, split=2, tokens=1024, exact_tail=0)
    rows = 700
    h = gen.normal((rows, cfg.d), 1.0, 3, "h", DEV, torch.bfloat16)
    layers = _layers_for(cfg, cfg.d, cfg.kvw, 2, 3, identity)
    shape = (2, 1, cfg.n_kv_heads, cfg.tokens, cfg.head_dim)
    x = {"h_split": h, "layers": layers,
         "k_cache": torch.full(shape, gen.CACHE_SENTINEL, dtype=torch.bfloat16, device=DEV),
         "v_cache": torch.full(shape, gen.CACHE_SENTINEL, dtype=torch.bfloat16, device=DEV)}
    f = _make(tee, cfg, layers, torch.bfloat16, cfg.tokens)
    f(h, x["k_cache"], x["v_cache"], pos0=100)
    _prefill_check(cfg, x, np.arange(0, rows, 7).astype(np.int64), rows, pos0=100)


def test_tc_fill_scattered_positions_sequences_and_device_count(tee):
    # A large batch of decode tokens: each row has its own sequence and position.
    cfg = configs.PrefillFillConfig(name="scatter", d=1024, n_layers=2, n_q_heads=8, n_kv_heads=4, head_dim=128,
                                    rope_base=1e4, split=0, tokens=2048, exact_tail=0)
    n_max, n = 600, 517
    h = gen.normal((n_max, cfg.d), 1.0, 5, "h", DEV, torch.bfloat16)
    layers = _layers_for(cfg, cfg.d, cfg.kvw, 2, 5)
    n_seq = 40
    # distinct (seq, pos) slots, so that no slot is written twice
    slots = torch.randperm(n_seq * cfg.tokens, generator=torch.Generator().manual_seed(5))[:n_max].to(DEV)
    seq, pos = (slots // cfg.tokens).int(), (slots % cfg.tokens).int()
    shape = (2, n_seq, cfg.n_kv_heads, cfg.tokens, cfg.head_dim)
    x = {"h_cur": h, "layers": layers,
         "k_cache": torch.full(shape, gen.CACHE_SENTINEL, dtype=torch.bfloat16, device=DEV),
         "v_cache": torch.full(shape, gen.CACHE_SENTINEL, dtype=torch.bfloat16, device=DEV)}
    f = _make(tee, cfg, layers, torch.bfloat16, cfg.tokens)
    n_dev = torch.tensor([n], dtype=torch.int32, device=DEV)
    f(h, x["k_cache"], x["v_cache"], pos=pos, seq=seq, n_dev=n_dev, n_max=n_max)
    cfg2 = configs.DecodeConfig(name="scatter", d=cfg.d, n_layers=2, n_q_heads=8, n_kv_heads=cfg.n_kv_heads,
                                head_dim=cfg.head_dim, batch=n_max, cache_len=cfg.tokens, gate_layer=0,
                                fill_layers=(0, 1), tau=0.5, rule="per_token", weights="dense", map="ridge",
                                rope_base=cfg.rope_base, dtype="bf16")
    check_decode_fill(cfg2, x, np.arange(n), pos.cpu().numpy(), seq.cpu().numpy(), gen.CACHE_SENTINEL)


def test_tc_fill_records_bad_positions(tee):
    cfg = configs.PREFILL_16K
    rows = 300
    x = gen.prefill_inputs(cfg, seed=4, device=DEV, rows=rows, layers=1)
    ws = tee.Workspace(DEV)
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.tokens)
    pos = torch.arange(rows, dtype=torch.int32, device=DEV)
    pos[17] = cfg.tokens + 3
    f(x["h_split"], x["k_cache"], x["v_cache"], pos=pos, ws=ws)
    code, detail = ws.device_error()
    assert code == 2 and detail == cfg.tokens + 3
    good = np.array([r for r in range(rows) if r != 17], dtype=np.int64)
    _prefill_check(cfg, {**x, "k_cache": x["k_cache"], "v_cache": x["v_cache"]}, good[::5], rows)
    assert bool((x["k_cache"][:, 0, :, 17] == gen.CACHE_SENTINEL).all())


def _sampled_rows(n, seed, k=48):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(16), np.arange(n - 16, n), rng.integers(0, n, k)])).astype(np.int64)


@pytest.mark.parametrize("cfg", [configs.PREFILL_16K, configs.PREFILL_120K], ids=["16k", "120k"])
def test_tc_fill_full_prefill_workload(tee, cfg):
    """The full workload in the launch configuration the bench times, checked on
    sampled rows (all layers) and, everywhere, on the slots that must stay untouched."""
    x = gen.prefill_inputs(cfg, seed=0, device=DEV)
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.tokens)
    f(x["h_split"], x["k_cache"], x["v_cache"])
    torch.cuda.synchronize()
    rows = _sampled_rows(cfg.filled_rows, 1)
    h = f64(x["h_split"][torch.as_tensor(rows, device=DEV)])
    for L in x["layers"]:
        Lh = host(L)
        k_ref, v_ref = oracle.fill_rows(h, Lh, rows, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps)
        j = L["cache_layer"]
        p = torch.as_tensor(rows, device=DEV)
        check_kv(x["k_cache"][j, 0].index_select(1, p).permute(1, 0, 2), k_ref, f"K layer {j}")
        check_kv(x["v_cache"][j, 0].index_select(1, p).permute(1, 0, 2), v_ref, f"V layer {j}")
        del Lh
    for c in (x["k_cache"], x["v_cache"]):
        assert bool((c[:, :, :, cfg.filled_rows:] == gen.CACHE_SENTINEL).all())   # exact tail untouched
        assert bool(torch.isfinite(c[:, :, :, :cfg.filled_rows]).all())
        assert not bool((c[:, :, :, :cfg.filled_rows] == gen.CACHE_SENTINEL).any())  # every filled slot written


# ---------------------------------------------------------------- decode path
# int4 fills of up to 128 items with an identity map run as one tcgen05 launch:
# one block per (64 output columns, layer), weights dequantised into the B operand.

@pytest.mark.parametrize("n,hd", [(1, 64), (17, 64), (100, 64), (128, 64), (48, 128)])
def test_decode_int4_fill_item_counts(tee, n, hd):
    base = configs.LLAMA1B_DECODE
    cfg = configs.DecodeConfig(**{**base.__dict__, "batch": n, "head_dim": hd, "n_kv_heads": 512 // hd})
    x = gen.decode_inputs(cfg, seed=n + hd, device=DEV, case="exit")
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.cache_len, int4=True)
    rng = np.random.default_rng(n)
    rows = rng.permutation(n).astype(np.int32)   # gathered in a scrambled order
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"])
    check_decode_fill(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL)


def test_decode_int4_fill_twice_reuses_the_workspace(tee):
    # the K-split partial tiles are cleared by the block that finishes each tile
    cfg = configs.LLAMA1B_DECODE
    ws = tee.Workspace(DEV)
    for seed in (7, 8):
        x = gen.decode_inputs(cfg, seed=seed, device=DEV, case="exit")
        f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.cache_len, int4=True)
        rows = np.arange(cfg.batch, dtype=np.int32)
        f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"],
          ws=ws)
        check_decode_fill(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL)
    assert ws.device_error() == (0, 0)


def test_decode_int4_fill_records_bad_positions(tee):
    cfg = configs.LLAMA1B_DECODE
    x = gen.decode_inputs(cfg, seed=9, device=DEV, case="exit")
    ws = tee.Workspace(DEV)
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.cache_len, int4=True)
    pos = x["pos"].clone()
    pos[5] = -1
    rows = torch.arange(cfg.batch, dtype=torch.int32, device=DEV)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=rows, pos=pos, seq=x["seq"], ws=ws)
    code, detail = ws.device_error()
    assert code == 2 and detail == -1
    good = np.array([r for r in range(cfg.batch) if r != 5], dtype=np.int32)
    check_decode_fill(cfg, x, good, pos.cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL)


# Shapes around the decode kernel's limits: d a multiple of 512 (one staged chunk of
# codes) takes the tcgen05 launch, fewer or more chunks than its four-chunk ring; other
# d go to the generic path. Same results either way.
@pytest.mark.parametrize("S,d,hd,n", [(8, 2048, 64, 64), (4, 1024, 128, 33), (1, 256, 64, 5), (3, 768, 64, 64),
                                      (8, 512, 128, 1), (2, 512, 64, 64), (2, 4096, 128, 128), (1, 5120, 128, 77),
                                      (2, 1536, 64, 100)])
def test_decode_shapes(tee, S, d, hd, n):
    base = configs.LLAMA1B_DECODE
    cfg = configs.DecodeConfig(**{**base.__dict__, "d": d, "batch": n, "head_dim": hd, "n_kv_heads": 512 // hd,
                                  "n_layers": S, "fill_layers": tuple(range(S))})
    x = gen.decode_inputs(cfg, seed=S * 100 + n, device=DEV, case="exit")
    f = _make(tee, cfg, x["layers"], torch.bfloat16, cfg.cache_len, int4=True)
    rows = np.random.default_rng(n).permutation(n).astype(np.int32)
    f(x["h_cur"], x["k_cache"], x["v_cache"], rows=torch.from_numpy(rows).to(DEV), pos=x["pos"], seq=x["seq"])
    check_decode_fill(cfg, x, rows, x["pos"].cpu().numpy(), x["seq"].cpu().numpy(), gen.CACHE_SENTINEL)
