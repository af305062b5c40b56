"""Cosine gate, compaction and exit scatter in one call (tee_exit_gate_compact_scatter)
on the GPU, against the oracle: scores within tolerance, everything the mask decides
bit-exact against the oracle's stable partition of the GPU's own mask."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import check_mask, check_scores, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def _states(n, d, dtype, seed, lo=0.8):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    hp = torch.randn(n, d, device=DEV, generator=g)
    a = lo + (1 - lo) * torch.rand(n, 1, device=DEV, generator=g)
    hc = a * hp + torch.sqrt(1 - a * a) * torch.randn(n, d, device=DEV, generator=g)
    return hp.to(dtype), hc.to(dtype)


def _check_all(res, out, out0, h_cur, pos_in, gather, s_ref, m_ref, tau, rule):
    check_scores(res["score"], s_ref)
    mask = res["mask"].cpu().numpy()
    if rule == "per_token":
        check_mask(res["mask"], s_ref, tau)
    elif np.abs(s_ref.min() - tau) > 1e-3:
        assert np.array_equal(mask, m_ref)
    # everything the GPU's mask decides is bit-exact
    part = oracle.stable_partition(mask, None if pos_in is None else pos_in.cpu().numpy())
    counts = res["counts"].cpu().numpy()
    assert list(counts) == list(part["counts"])
    nc, ne = counts
    for k, m in (("cont_rows", nc), ("exit_rows", ne), ("cont_pos", nc), ("exit_pos", ne)):
        assert np.array_equal(res[k].cpu().numpy()[:m], part[k]), k
    # the flag: every token's score (as the GPU computed it, in fp32) above tau
    assert int(res["flag"].item()) == int(bool((res["score"] > tau).all().item()))
    if gather:
        assert torch.equal(res["h_cont"][:nc].cpu(), h_cur.cpu()[torch.from_numpy(part["cont_rows"]).long()])
    want = oracle.exit_scatter(f64(out0), f64(h_cur), part["exit_rows"], part["exit_pos"])
    assert np.array_equal(f64(out), want)


@pytest.mark.parametrize("n", [1, 5, 16, 17, 64, 100, 128, 129, 300])
@pytest.mark.parametrize("d,dtype", [(2048, torch.bfloat16), (4096, torch.bfloat16), (256, torch.float32),
                                     (520, torch.float16)])
@pytest.mark.parametrize("rule", ["per_token", "batch_all"])
def test_gate_compact_scatter(tee, n, d, dtype, rule):
    tau = 0.9 if rule == "per_token" else 0.75
    hp, hc = _states(n, d, dtype, seed=n * 7 + d)
    rng = np.random.default_rng(n + d)
    pos_in = torch.from_numpy(rng.permutation(2 * n)[:n].astype(np.int32)).to(DEV) if n % 2 else None
    n_out = 2 * n
    out0 = torch.full((n_out, d), -5.0, device=DEV).to(dtype)
    out = out0.clone()
    gather = n % 3 != 0
    ws = tee.Workspace(DEV)
    res = tee.exit_gate_compact_scatter(hc, hp, tau, out, rule=rule, pos_in=pos_in, gather=gather, ws=ws)
    torch.cuda.synchronize()
    assert ws.device_error() == (0, 0)
    s_ref, m_ref, f_ref = oracle.cosine_gate(f64(hp), f64(hc), tau, rule)
    _check_all(res, out, out0, hc, pos_in, gather, s_ref, m_ref, tau, rule)


def test_gate_compact_scatter_batch_cases(tee):
    # batch rule at decode size: every token exits (tau below all scores) or none (one low score)
    n, d = 64, 2048
    hp, hc = _states(n, d, torch.bfloat16, seed=1, lo=0.99)
    for tau, expect in ((0.95, 1), (0.99999, 0)):
        out = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)
        res = tee.exit_gate_compact_scatter(hc, hp, tau, out, rule="batch_all")
        torch.cuda.synchronize()
        assert int(res["flag"].item()) == expect
        assert int(res["counts"][1].item()) == expect * n
        assert bool((res["mask"] == expect).all())
        if expect:
            assert torch.equal(out, hc)
        else:
            assert torch.equal(res["h_cont"], hc)


def test_gate_compact_scatter_matches_the_separate_calls(tee):
    n, d = 64, 2048
    hp, hc = _states(n, d, torch.bfloat16, seed=3)
    out1 = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)
    out2 = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)
    score, mask, flag = tee.exit_gate(hc, 0.9, h_prev=hp)
    r1 = tee.exit_compact_scatter(mask, hc, out1)
    r2 = tee.exit_gate_compact_scatter(hc, hp, 0.9, out2)
    torch.cuda.synchronize()
    assert (score - r2["score"]).abs().max().item() <= 1e-5
    if bool(torch.equal(mask, r2["mask"])):
        assert torch.equal(out1, out2)
        for k in ("counts", "exit_rows"):
            assert torch.equal(r1[k][:int(r1["counts"][1]) if k != "counts" else 2],
                               r2[k][:int(r2["counts"][1]) if k != "counts" else 2])


def test_gate_compact_scatter_records_bad_slots(tee):
    n, d = 40, 256
    hp, hc = _states(n, d, torch.bfloat16, seed=9, lo=0.999)
    pos_in = torch.arange(n, dtype=torch.int32, device=DEV)
    pos_in[3] = n + 5
    out = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)
    ws = tee.Workspace(DEV)
    res = tee.exit_gate_compact_scatter(hc, hp, 0.5, out, pos_in=pos_in, ws=ws)
    torch.cuda.synchronize()
    assert int(res["counts"][1].item()) == n
    assert ws.device_error() == (5, n + 5)
    keep = [i for i in range(n) if i != 3]
    assert torch.equal(out[keep], hc[keep])
    assert bool((out[3] == 0).all())


def test_gate_compact_scatter_empty(tee):
    hp = torch.zeros(0, 256, device=DEV, dtype=torch.bfloat16)
    out = torch.zeros(4, 256, device=DEV, dtype=torch.bfloat16)
    res = tee.exit_gate_compact_scatter(hp, hp, 0.5, out)
    torch.cuda.synchronize()
    assert res["counts"].tolist() == [0, 0]
