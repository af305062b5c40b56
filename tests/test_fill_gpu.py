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
