"""A whole decode step on the GPU - gate, compaction, KV fill, exit scatter -
chained on the device (counts never leave the GPU), against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import NEAR_BAND, check_decode_fill, check_mask, check_scores, f64
from workloads import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def run_step(tee, cfg, x, fill, ws, scatter_first=False, fused=False):
    out = torch.full_like(x["h_cur"], -3.0)
    if fused == "front":   # gate, compaction and scatter in one launch, then the fill
        comp = tee.exit_gate_compact_scatter(x["h_cur"], x["h_prev"], cfg.tau, out, rule=cfg.rule, ws=ws)
        fill(x["h_cur"], x["k_cache"], x["v_cache"], rows=comp["exit_rows"], pos=x["pos"], seq=x["seq"],
             n_dev=comp["counts"][1:], n_max=cfg.batch, ws=ws)
        return comp["score"], comp["mask"], comp["flag"], comp, out
    score, mask, flag = tee.exit_gate(x["h_cur"], cfg.tau, h_prev=x["h_prev"], rule=cfg.rule, ws=ws)
    if fused:   # compaction and scatter in one launch, then the fill
        comp = tee.exit_compact_scatter(mask, x["h_cur"], out, ws=ws)
        fill(x["h_cur"], x["k_cache"], x["v_cache"], rows=comp["exit_rows"], pos=x["pos"], seq=x["seq"],
             n_dev=comp["counts"][1:], n_max=cfg.batch, ws=ws)
        return score, mask, flag, comp, out
    comp = tee.exit_compact(mask, h=x["h_cur"], ws=ws)

    def do_fill():
        fill(x["h_cur"], x["k_cache"], x["v_cache"], rows=comp["exit_rows"], pos=x["pos"], seq=x["seq"],
             n_dev=comp["counts"][1:], n_max=cfg.batch, ws=ws)

    def do_scatter():
        tee.exit_scatter(comp["counts"], comp["exit_rows"], comp["exit_pos"], x["h_cur"], out, ws=ws)

    if scatter_first:   # the fill then follows the scatter kernel directly (early launch)
        do_scatter()
        do_fill()
    else:
        do_fill()
        do_scatter()
    return score, mask, flag, comp, out


@pytest.mark.parametrize("cfg,case,seed,early,fused",
                         [(configs.TINY_DECODE, "default", s, False, False) for s in range(4)] +
                         [(configs.TINY_DECODE, "default", s, False, True) for s in range(2)] +
                         [(configs.LLAMA1B_DECODE, c, s, False, False) for c in ("exit", "stay") for s in range(2)] +
                         [(configs.LLAMA1B_DECODE, c, s, True, False) for c in ("exit", "stay") for s in range(2)] +
                         [(configs.LLAMA1B_DECODE, c, s, True, True) for c in ("exit", "stay") for s in range(2)] +
                         [(configs.TINY_DECODE, "default", s, False, "front") for s in range(4)] +
                         [(configs.LLAMA1B_DECODE, c, s, True, "front") for c in ("exit", "stay") for s in range(2)])
def test_decode_step(tee, cfg, case, seed, early, fused, record_property):
    # early: the fill launches while the previous kernel runs and reads h, rows, counts
    # only after it completes (TEE_FILL_EARLY_WEIGHTS); fused: compaction and scatter
    # in one launch; "front": gate, compaction and scatter in one launch (the bench's step)
    x = gen.decode_inputs(cfg, seed=seed, device=DEV, case=case)
    ws = tee.Workspace(DEV)
    fill = tee.KVFill(x["layers"], d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                      rope_base=cfg.rope_base, eps=cfg.eps, dtype=x["h_cur"].dtype, max_pos=cfg.cache_len,
                      int4=cfg.weights == "int4", group=cfg.group, early_weights=early)
    score, mask, flag, comp, out = run_step(tee, cfg, x, fill, ws, scatter_first=early, fused=fused)
    assert ws.device_error() == (0, 0)
    hp, hc = f64(x["h_prev"]), f64(x["h_cur"])
    s_ref, m_ref, f_ref = oracle.cosine_gate(hp, hc, cfg.tau, cfg.rule)
    check_scores(score, s_ref)
    # Exit decisions: bit-exact except tokens whose score lies within 1e-3 of tau,
    # which are excluded and counted. Under the batch-min rule every token takes the
    # one decision of the lowest score, so that decision is excluded when the lowest
    # score is in the band.
    gpu_mask = mask.cpu().numpy()
    if cfg.rule == "batch_all":
        near = abs(float(s_ref.min()) - cfg.tau) <= NEAR_BAND
        excluded = cfg.batch if near else 0
        if not near:
            assert int(flag.item()) == f_ref and np.array_equal(gpu_mask, m_ref)
        assert np.all(gpu_mask == gpu_mask[0]) and int(flag.item()) == int(gpu_mask[0])
    else:
        excluded = check_mask(mask, s_ref, cfg.tau)
        if excluded == 0:
            assert np.array_equal(gpu_mask, m_ref)
    record_property("excluded_near_threshold", excluded)
    # Compaction, fill and scatter follow the GPU's own decisions, with no exclusion:
    # bit-exact partition and scatter, the fill within the K/V bound.
    part = oracle.stable_partition(gpu_mask)
    counts = comp["counts"].cpu().numpy()
    assert list(counts) == list(part["counts"])
    assert np.array_equal(comp["exit_rows"].cpu().numpy()[:counts[1]], part["exit_rows"])
    assert torch.equal(comp["h_cont"][:counts[0]].cpu(), x["h_cur"].cpu()[torch.from_numpy(part["cont_rows"]).long()])
    pos, seq = x["pos"].cpu().numpy(), x["seq"].cpu().numpy()
    check_decode_fill(cfg, x, part["exit_rows"], pos, seq, gen.CACHE_SENTINEL)
    o_ref = oracle.exit_scatter(np.full(hc.shape, -3.0), hc, part["exit_rows"], part["exit_pos"])
    assert np.array_equal(f64(out), o_ref)


@pytest.mark.parametrize("cfg,case,seed", [(configs.TINY_DECODE, "default", 0), (configs.TINY_DECODE, "default", 3),
                                           (configs.LLAMA1B_DECODE, "exit", 0), (configs.LLAMA1B_DECODE, "stay", 1)])
def test_decode_step_from_host_buffers(tee, cfg, case, seed):
    """tee_decode_step_run_host (host inputs copied in, front and fill, results copied
    out, one call) gives exactly what the two device calls give on the same inputs."""
    x = gen.decode_inputs(cfg, seed=seed, device=DEV, case=case)
    dt = x["h_cur"].dtype
    mk = lambda: tee.KVFill(x["layers"], d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,  # noqa: E731
                            rope_base=cfg.rope_base, eps=cfg.eps, dtype=dt, max_pos=cfg.cache_len,
                            int4=cfg.weights == "int4", group=cfg.group)
    # device path on its own copies of the caches
    k_dev, v_dev = x["k_cache"].clone(), x["v_cache"].clone()
    ws = tee.Workspace(DEV)
    out_dev = torch.zeros_like(x["h_cur"])
    comp = tee.exit_gate_compact_scatter(x["h_cur"], x["h_prev"], cfg.tau, out_dev, rule=cfg.rule, ws=ws)
    mk()(x["h_cur"], k_dev, v_dev, rows=comp["exit_rows"], pos=x["pos"], seq=x["seq"], n_dev=comp["counts"][1:],
         n_max=cfg.batch, ws=ws)
    # the one-call path from pinned host buffers
    step = tee.DecodeStep(mk(), n_max=cfg.batch, d=cfg.d, threshold=cfg.tau, dtype=dt, rule=cfg.rule,
                          k_cache=x["k_cache"], v_cache=x["v_cache"])
    hi = {k: x[k].cpu().pin_memory() for k in ("h_prev", "h_cur", "pos", "seq")}
    score = torch.empty(cfg.batch).pin_memory()
    mask = torch.empty(cfg.batch, dtype=torch.uint8).pin_memory()
    counts = torch.empty(2, dtype=torch.int32).pin_memory()
    out = torch.empty(cfg.batch, cfg.d, dtype=dt).pin_memory()
    step.run_host(hi["h_prev"], hi["h_cur"], hi["pos"], hi["seq"], score=score, mask=mask, counts=counts, out=out)
    torch.cuda.synchronize()
    assert step.ws.device_error() == (0, 0) and ws.device_error() == (0, 0)
    assert torch.equal(score, comp["score"].cpu()) and torch.equal(mask, comp["mask"].cpu())
    assert torch.equal(counts, comp["counts"].cpu())
    n_exit = int(counts[1])
    rows = comp["exit_rows"][:n_exit].long()
    assert torch.equal(out[rows.cpu()], out_dev[rows].cpu())   # the exiting rows, scattered to their slots
    assert torch.equal(x["k_cache"], k_dev) and torch.equal(x["v_cache"], v_dev)
    # again with the same host buffers (the captured step replayed), then from pageable
    # host memory (no capture: the calls enqueued directly); the same results each time
    for host in (hi, {k: t.clone() for k, t in hi.items()}):
        score2, mask2, counts2, out2 = score.clone().zero_(), mask.clone().zero_(), counts.clone().zero_(), out.clone()
        if host is hi:
            score2, mask2, counts2, out2 = score2.pin_memory(), mask2.pin_memory(), counts2.pin_memory(), out2.pin_memory()
        step.run_host(host["h_prev"], host["h_cur"], host["pos"], host["seq"], score=score2, mask=mask2,
                      counts=counts2, out=out2)
        torch.cuda.synchronize()
        assert torch.equal(score2, score) and torch.equal(mask2, mask) and torch.equal(counts2, counts)
        assert torch.equal(out2[rows.cpu()], out[rows.cpu()])
        assert torch.equal(x["k_cache"], k_dev) and torch.equal(x["v_cache"], v_dev)


@pytest.mark.parametrize("cfg", [configs.TINY_DECODE, configs.LLAMA1B_DECODE])
def test_decode_step_replays_read_the_rewritten_host_buffers(tee, cfg):
    """A serving loop rewrites the same pinned host buffers every step and the
    captured step is replayed on them: each replay must see that step's inputs
    (the copies run in the replay, and nothing is served from a cache), equal to
    the device calls on the same inputs."""
    x = gen.decode_inputs(cfg, seed=11, device=DEV, case="default")
    dt = x["h_cur"].dtype
    mk = lambda: tee.KVFill(x["layers"], d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,  # noqa: E731
                            rope_base=cfg.rope_base, eps=cfg.eps, dtype=dt, max_pos=cfg.cache_len,
                            int4=cfg.weights == "int4", group=cfg.group)
    step = tee.DecodeStep(mk(), n_max=cfg.batch, d=cfg.d, threshold=cfg.tau, dtype=dt, rule=cfg.rule,
                          k_cache=x["k_cache"], v_cache=x["v_cache"])
    hi = {k: x[k].cpu().pin_memory() for k in ("h_prev", "h_cur", "pos", "seq")}
    score = torch.empty(cfg.batch).pin_memory()
    mask = torch.empty(cfg.batch, dtype=torch.uint8).pin_memory()
    counts = torch.empty(2, dtype=torch.int32).pin_memory()
    out = torch.empty(cfg.batch, cfg.d, dtype=dt).pin_memory()
    fill, ws = mk(), tee.Workspace(DEV)
    for seed in (11, 12, 13):
        y = gen.decode_inputs(cfg, seed=seed, device=DEV, case="default")
        for k in hi:   # this step's inputs, written in place into the same host buffers
            hi[k].copy_(y[k].cpu())
        k_dev, v_dev = x["k_cache"].clone(), x["v_cache"].clone()   # the caches before this step
        out.fill_(-3.0)
        step.run_host(hi["h_prev"], hi["h_cur"], hi["pos"], hi["seq"], score=score, mask=mask, counts=counts, out=out)
        out_dev = torch.full_like(y["h_cur"], -3.0)
        comp = tee.exit_gate_compact_scatter(y["h_cur"], y["h_prev"], cfg.tau, out_dev, rule=cfg.rule, ws=ws)
        fill(y["h_cur"], k_dev, v_dev, rows=comp["exit_rows"], pos=y["pos"], seq=y["seq"], n_dev=comp["counts"][1:],
             n_max=cfg.batch, ws=ws)
        torch.cuda.synchronize()
        assert step.ws.device_error() == (0, 0) and ws.device_error() == (0, 0)
        assert torch.equal(score, comp["score"].cpu()) and torch.equal(mask, comp["mask"].cpu())
        assert torch.equal(counts, comp["counts"].cpu())
        rows = comp["exit_rows"][:int(counts[1])].long()
        assert torch.equal(out[rows.cpu()], out_dev[rows].cpu())
        assert torch.equal(x["k_cache"], k_dev) and torch.equal(x["v_cache"], v_dev)
