"""Compaction and exit scatter on the GPU against the brute-force oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import f64
from workloads import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def _masks(n, rng):
    yield "none", np.zeros(n, np.uint8)
    yield "all", np.ones(n, np.uint8)
    yield "alternating", (np.arange(n) % 2).astype(np.uint8)
    yield "random", (rng.random(n) < 0.37).astype(np.uint8) * rng.integers(1, 256, n).astype(np.uint8)


def _check(res, ref, n, h=None):
    counts = res["counts"].cpu().numpy()
    assert list(counts) == list(ref["counts"])
    nc, ne = counts
    for k, m in (("cont_rows", nc), ("exit_rows", ne), ("cont_pos", nc), ("exit_pos", ne)):
        if k in res:
            assert np.array_equal(res[k].cpu().numpy()[:m], ref[k]), k
    if h is not None:
        assert torch.equal(res["h_cont"][:nc].cpu(), h.cpu()[torch.from_numpy(ref["cont_rows"]).long()])


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 64, 255, 256, 257, 4095, 4096, 4097, 65536, 65537, 200003])
def test_compaction_indices(tee, n):
    rng = np.random.default_rng(n)
    pos_in = torch.from_numpy(rng.permutation(10 * n)[:n].astype(np.int32)).to(DEV)
    for name, m in _masks(n, rng):
        mask = torch.from_numpy(m).to(DEV)
        res = tee.exit_compact(mask, pos_in=pos_in)
        _check(res, oracle.stable_partition(m, pos_in.cpu().numpy()), n)


@pytest.mark.parametrize("n,d,dtype", [(32, 4096, torch.bfloat16), (4096, 4096, torch.bfloat16),
                                       (33, 256, torch.float32), (1000, 520, torch.float16),
                                       (70000, 64, torch.bfloat16)])
def test_compaction_with_gather(tee, n, d, dtype):
    rng = np.random.default_rng(d + n)
    h = torch.randn(n, d, device=DEV).to(dtype)
    for name, m in _masks(n, rng):
        res = tee.exit_compact(torch.from_numpy(m).to(DEV), h=h)
        _check(res, oracle.stable_partition(m), n, h)


def test_compaction_empty(tee):
    res = tee.exit_compact(torch.empty(0, dtype=torch.uint8, device=DEV))
    assert res["counts"].tolist() == [0, 0]


def test_compaction_fed_by_the_gpu_gate(tee):
    # No exclusions: compaction must follow the GPU's own mask exactly.
    cfg = configs.ROUTER_4096
    w = gen.router_weights(cfg, 3, seed=0, device=DEV)
    h = gen.router_hidden(cfg, 4096, 3, seed=0, device=DEV)
    _, mask, _ = tee.exit_gate(h, 0.5, w_down=w["w_down"], w_up=w["w_up"])
    res = tee.exit_compact(mask, h=h)
    _check(res, oracle.stable_partition(mask.cpu().numpy()), 4096, h)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n", [8, 64, 4096])
def test_scatter_restores_exiting_rows(tee, n, dtype):
    d = 1024 if n < 4096 else 4096
    rng = np.random.default_rng(n)
    h = torch.randn(n, d, device=DEV).to(dtype)
    m = (rng.random(n) < 0.5).astype(np.uint8)
    orig = torch.from_numpy(rng.permutation(3 * n)[:n].astype(np.int32)).to(DEV)
    res = tee.exit_compact(torch.from_numpy(m).to(DEV), pos_in=orig)
    out = torch.full((3 * n, d), -7.0, device=DEV, dtype=dtype)
    tee.exit_scatter(res["counts"], res["exit_rows"], res["exit_pos"], h, out)
    ref = oracle.exit_scatter(np.full((3 * n, d), -7.0), f64(h), *[oracle.stable_partition(m, orig.cpu().numpy())[k]
                                                                   for k in ("exit_rows", "exit_pos")])
    assert np.array_equal(f64(out), ref)


def test_exit_projection_rmsnorm_scatter(tee):
    n, d = 300, 2048
    h = torch.randn(n, d, device=DEV, dtype=torch.bfloat16) * 3
    gamma = (1 + 0.1 * torch.randn(d, device=DEV)).bfloat16()
    m = (np.arange(n) % 3 == 0).astype(np.uint8)
    res = tee.exit_compact(torch.from_numpy(m).to(DEV))
    out = torch.zeros(n, d, device=DEV, dtype=torch.float32)
    hf = h.float()
    tee.exit_scatter(res["counts"], res["exit_rows"], res["exit_rows"], hf, out, final_gamma=gamma.float(), eps=1e-5)
    part = oracle.stable_partition(m)
    ref = oracle.exit_scatter(np.zeros((n, d)), f64(hf), part["exit_rows"], part["exit_rows"], gamma=f64(gamma),
                              eps=1e-5)
    assert np.abs(f64(out) - ref).max() < 1e-4


def test_scatter_records_bad_destinations(tee):
    n, d = 16, 64
    ws = tee.Workspace(DEV)
    h = torch.randn(n, d, device=DEV)
    counts = torch.tensor([0, 3], dtype=torch.int32, device=DEV)
    rows = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    dest = torch.tensor([5, 99, 6], dtype=torch.int32, device=DEV)   # 99 is outside out
    out = torch.zeros(8, d, device=DEV)
    tee.exit_scatter(counts, rows, dest, h, out, ws=ws)
    code, detail = ws.device_error()
    assert code == 5 and detail == 99  # TEE_DEVERR_DEST
    assert torch.equal(out[5], h[0]) and torch.equal(out[6], h[2])
    ws.clear_error()
    assert ws.device_error() == (0, 0)


# ------------------------------------------------------------ compaction + scatter in one launch

@pytest.mark.parametrize("n,d,dtype,gather", [(1, 256, torch.bfloat16, True), (8, 2048, torch.bfloat16, False),
                                              (33, 256, torch.float32, True), (64, 2048, torch.bfloat16, True),
                                              (300, 520, torch.float16, False), (4097, 256, torch.bfloat16, True),
                                              (70000, 64, torch.bfloat16, True)])
def test_compaction_with_scatter(tee, n, d, dtype, gather):
    rng = np.random.default_rng(n + d)
    h = torch.randn(n, d, device=DEV).to(dtype)
    n_out = 3 * n
    pos_in = torch.from_numpy(rng.permutation(n_out)[:n].astype(np.int32)).to(DEV)
    for name, m in _masks(n, rng):
        out = torch.full((n_out, d), -7.0, device=DEV).to(dtype)
        ws = tee.Workspace(DEV)
        res = tee.exit_compact_scatter(torch.from_numpy(m).to(DEV), h, out, pos_in=pos_in, gather=gather, ws=ws)
        ref = oracle.stable_partition(m, pos_in.cpu().numpy())
        _check(res, ref, n, h if gather else None)
        want = oracle.exit_scatter(np.full((n_out, d), -7.0), f64(h), ref["exit_rows"], ref["exit_pos"])
        assert torch.equal(out.cpu(), torch.from_numpy(want).to(dtype)), name
        assert ws.device_error() == (0, 0)


def test_compaction_with_scatter_matches_the_two_calls(tee):
    # the decode-step shape: 64 tokens of a 1B model, identity slots
    n, d = 64, 2048
    h = torch.randn(n, d, device=DEV).to(torch.bfloat16)
    m = torch.from_numpy((np.random.default_rng(3).random(n) < 0.5).astype(np.uint8)).to(DEV)
    out1 = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)
    out2 = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)
    r1 = tee.exit_compact(m, h=h)
    tee.exit_scatter(r1["counts"], r1["exit_rows"], r1["exit_pos"], h, out1)
    r2 = tee.exit_compact_scatter(m, h, out2)
    assert torch.equal(out1, out2)
    for k in ("counts", "cont_rows", "exit_rows", "h_cont"):
        c = int(r1["counts"][0]) if k in ("cont_rows", "h_cont") else int(r1["counts"][1]) if k == "exit_rows" else 2
        assert torch.equal(r1[k][:c], r2[k][:c]), k


def test_compaction_with_scatter_records_bad_slots(tee):
    n, d = 40, 256
    h = torch.randn(n, d, device=DEV).to(torch.bfloat16)
    m = torch.ones(n, dtype=torch.uint8, device=DEV)
    pos_in = torch.arange(n, dtype=torch.int32, device=DEV)
    pos_in[5] = n + 3     # outside out's rows: skipped and recorded
    pos_in[9] = -1
    out = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)
    ws = tee.Workspace(DEV)
    tee.exit_compact_scatter(m, h, out, pos_in=pos_in, gather=False, ws=ws)
    code, detail = ws.device_error()
    assert code == 5 and detail in (n + 3, -1)
    keep = [i for i in range(n) if i not in (5, 9)]
    assert torch.equal(out[keep], h[keep])
    assert torch.equal(out[5], torch.zeros(d, device=DEV, dtype=torch.bfloat16))
    assert torch.equal(out[9], torch.zeros(d, device=DEV, dtype=torch.bfloat16))
