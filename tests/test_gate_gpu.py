"""Exit gate on the GPU (through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import check_mask, check_scores, f64
from workloads import configs, gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


DEV = "cuda"


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cosine_tiny_fp32_per_token(tee, seed):
    cfg = configs.TINY_DECODE
    x = gen.decode_inputs(cfg, seed=seed, device=DEV, with_cache=False)
    score, mask, flag = tee.exit_gate(x["h_cur"], cfg.tau, h_prev=x["h_prev"], rule="per_token")
    s_ref, m_ref, f_ref = oracle.cosine_gate(f64(x["h_prev"]), f64(x["h_cur"]), cfg.tau, "per_token")
    check_scores(score, s_ref)
    check_mask(mask, s_ref, cfg.tau)
    if np.all(np.abs(s_ref - cfg.tau) > 1e-3):
        assert int(flag.item()) == f_ref


@pytest.mark.parametrize("case,want", [("exit", 1), ("stay", 0)])
@pytest.mark.parametrize("seed", [0, 1])
def test_cosine_bf16_batch_min(tee, case, want, seed):
    cfg = configs.LLAMA1B_DECODE
    x = gen.decode_inputs(cfg, seed=seed, device=DEV, case=case, with_cache=False)
    score, mask, flag = tee.exit_gate(x["h_cur"], cfg.tau, h_prev=x["h_prev"], rule="batch_all")
    s_ref, m_ref, f_ref = oracle.cosine_gate(f64(x["h_prev"]), f64(x["h_cur"]), cfg.tau, "batch_all")
    check_scores(score, s_ref)
    assert f_ref == want and int(flag.item()) == want
    assert np.array_equal(mask.cpu().numpy(), m_ref)


@pytest.mark.parametrize("n", [1, 7, 31, 32, 33, 255, 4095, 4096, 4097, 9000])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_cosine_sizes_and_dtypes(tee, n, dtype):
    cfg = configs.DecodeConfig(**{**configs.TINY_DECODE.__dict__, "batch": n, "d": 264})
    x = gen.decode_inputs(cfg, seed=n, device=DEV, with_cache=False)
    hp, hc = x["h_prev"].to(dtype), x["h_cur"].to(dtype)
    for rule in ("per_token", "batch_all"):
        score, mask, flag = tee.exit_gate(hc, 0.9, h_prev=hp, rule=rule)
        s_ref, m_ref, f_ref = oracle.cosine_gate(f64(hp), f64(hc), 0.9, rule)
        check_scores(score, s_ref)
        if rule == "per_token":
            check_mask(mask, s_ref, 0.9)
        elif np.abs(s_ref.min() - 0.9) > 1e-3:
            assert int(flag.item()) == f_ref and np.array_equal(mask.cpu().numpy(), m_ref)


def test_cosine_strided_rows_and_zero_rows(tee):
    base = torch.randn(40, 512, device=DEV, dtype=torch.bfloat16)
    hp, hc = base[:, :256], base[:, 256:]           # ld = 512
    hp[3].zero_()
    score, mask, flag = tee.exit_gate(hc, -0.5, h_prev=hp)
    s_ref, _, _ = oracle.cosine_gate(f64(hp), f64(hc), -0.5)
    check_scores(score, s_ref)
    assert float(score[3]) == 0.0 and int(mask[3]) == 1   # 0 > -0.5


def test_gate_empty_batch(tee):
    h = torch.empty(0, 256, device=DEV)
    score, mask, flag = tee.exit_gate(h, 0.5, h_prev=h, rule="batch_all")
    assert int(flag.item()) == 0 and score.numel() == 0


def _router_ref(h, w, theta, rule, **kw):
    return oracle.router_gate(f64(h), f64(w["w_down"]), f64(w["w_up"]), theta, rule,
                              **{k: (f64(v) if torch.is_tensor(v) else v) for k, v in kw.items()})


@pytest.mark.parametrize("n", [32, 4096])
@pytest.mark.parametrize("theta", configs.ROUTER_4096.thetas)
def test_router_workload(tee, n, theta):
    cfg = configs.ROUTER_4096
    k = cfg.checkpoints[n % len(cfg.checkpoints)]
    w = gen.router_weights(cfg, k, seed=0, device=DEV)
    h = gen.router_hidden(cfg, n, k, seed=0, device=DEV)
    score, mask, flag = tee.exit_gate(h, theta, w_down=w["w_down"], w_up=w["w_up"], eps=cfg.eps)
    p_ref, m_ref, _ = _router_ref(h, w, theta, "per_token", eps=cfg.eps)
    check_scores(score, p_ref)
    excluded = check_mask(mask, p_ref, theta)
    assert excluded <= max(2, n // 20)


@pytest.mark.parametrize("n", [1, 5, 33, 300])
def test_router_biases_gamma_and_batch_rule(tee, n):
    cfg = configs.ROUTER_4096
    d = 1024
    torch.manual_seed(n)
    h = torch.randn(n, d, device=DEV, dtype=torch.bfloat16)
    w = {"w_down": (0.02 * torch.randn(128, d, device=DEV)).bfloat16(),
         "w_up": (0.02 * torch.randn(128, device=DEV)).bfloat16()}
    gamma = (1 + 0.1 * torch.randn(d, device=DEV)).bfloat16()
    b_down = 0.1 * torch.randn(128, device=DEV)
    b_up = torch.tensor([2.0], device=DEV)  # p well above 0.5 for every token
    for rule in ("per_token", "batch_all"):
        score, mask, flag = tee.exit_gate(h, 0.6, w_down=w["w_down"], w_up=w["w_up"], gamma=gamma, b_down=b_down,
                                          b_up=b_up, rule=rule, eps=cfg.eps)
        p_ref, m_ref, f_ref = _router_ref(h, w, 0.6, rule, gamma=gamma, b_down=b_down, b_up=b_up, eps=cfg.eps)
        check_scores(score, p_ref)
        assert int(flag.item()) == f_ref == 1
        assert np.array_equal(mask.cpu().numpy(), m_ref)


def test_router_zero_weights_give_sigmoid_bias(tee):
    n, d = 64, 512
    h = torch.randn(n, d, device=DEV, dtype=torch.bfloat16)
    z = torch.zeros(128, d, device=DEV, dtype=torch.bfloat16)
    score, _, _ = tee.exit_gate(h, 0.5, w_down=z, w_up=torch.zeros(128, device=DEV, dtype=torch.bfloat16),
                                b_up=torch.tensor([np.log(3.0)], device=DEV, dtype=torch.float32))
    assert torch.allclose(score, torch.full_like(score, 0.75), atol=1e-6)


# ------------------------------------------------------------ router on tcgen05
# bf16 batches of at least 256 tokens without gamma run the d -> 128 contraction
# on the tensor cores (K split across CTAs, partial sums accumulated in the workspace).

@pytest.mark.parametrize("n", [256, 300, 1000, 8192])
def test_router_tc_batch_sizes(tee, n):
    cfg = configs.ROUTER_4096
    w = gen.router_weights(cfg, 7, seed=n, device=DEV)
    h = gen.router_hidden(cfg, n, 7, seed=n, device=DEV)
    b_down = 0.05 * torch.randn(128, device=DEV)
    score, mask, flag = tee.exit_gate(h, 0.5, w_down=w["w_down"], w_up=w["w_up"], b_down=b_down, eps=cfg.eps)
    p_ref, _, _ = _router_ref(h, w, 0.5, "per_token", b_down=b_down, eps=cfg.eps)
    check_scores(score, p_ref)
    check_mask(mask, p_ref, 0.5)


# Above 76 token tiles (on 152 SMs) the gate runs one persistent CTA per SM over
# the tiles, two TMEM accumulators, no K split: 9729 tokens = 77 tiles with a
# one-token tail; 40000 tokens = 313 tiles, two or three per CTA, a 64-token tail.
@pytest.mark.parametrize("n,rule", [(9729, "per_token"), (40000, "per_token"), (40000, "batch_all")])
def test_router_tc_persistent(tee, n, rule):
    cfg = configs.ROUTER_4096
    w = gen.router_weights(cfg, 3, seed=n, device=DEV)
    h = gen.router_hidden(cfg, n, 3, seed=n, device=DEV)
    b_down = 0.05 * torch.randn(128, device=DEV)
    b_up = torch.full((1,), 0.3, device=DEV)
    ws = tee.Workspace(DEV)
    score, mask, flag = tee.exit_gate(h, 0.5, w_down=w["w_down"], w_up=w["w_up"], b_down=b_down, b_up=b_up,
                                      rule=rule, eps=cfg.eps, ws=ws)
    p_ref, m_ref, f_ref = _router_ref(h, w, 0.5, rule, b_down=b_down, b_up=b_up, eps=cfg.eps)
    check_scores(score, p_ref)
    if rule == "per_token":
        check_mask(mask, p_ref, 0.5)
    elif np.abs(p_ref.min() - 0.5) > 1e-3:
        assert int(flag.item()) == int(f_ref)
        assert bool((mask == int(f_ref)).all())
    assert ws.device_error() == (0, 0)


# d that is not a whole number of two-block stages (the trailing block reads as
# zero), with the K split (4096 tokens) and the persistent kernel (20000 tokens).
@pytest.mark.parametrize("d,n", [(576, 4096), (576, 20000), (64, 300), (192, 9729)])
def test_router_tc_odd_k_blocks(tee, d, n):
    import dataclasses
    cfg = dataclasses.replace(configs.ROUTER_4096, d=d)
    w = gen.router_weights(cfg, 1, seed=d, device=DEV)
    w["w_down"] = (w["w_down"].float() * 6.0).to(torch.bfloat16)   # keep the scores spread at small d
    h = gen.router_hidden(cfg, n, 1, seed=d, device=DEV)
    b_down = 0.05 * torch.randn(128, device=DEV)
    score, mask, _ = tee.exit_gate(h, 0.5, w_down=w["w_down"], w_up=w["w_up"], b_down=b_down, eps=cfg.eps)
    p_ref, _, _ = _router_ref(h, w, 0.5, "per_token", b_down=b_down, eps=cfg.eps)
    check_scores(score, p_ref)
    check_mask(mask, p_ref, 0.5)


def test_router_tc_persistent_on_the_exact_workspace(tee):
    # The persistent kernel needs no scratch beyond the header: the call runs on a
    # buffer of exactly the queried size, through the C ABI.
    import ctypes
    from token_early_exit_gb300 import _lib
    cfg = configs.ROUTER_4096
    n = 20000
    w = gen.router_weights(cfg, 7, seed=5, device=DEV)
    h = gen.router_hidden(cfg, n, 7, seed=5, device=DEV)
    lib = _lib.load()
    desc = _lib.GateDesc(mode=_lib.TEE_GATE_ROUTER, rule=_lib.TEE_RULE_PER_TOKEN, dtype=_lib.TEE_BF16, d=cfg.d,
                         bottleneck=cfg.bottleneck, threshold=0.5, eps=cfg.eps)
    size = lib.tee_exit_gate_workspace_size(ctypes.byref(desc), n)
    ws = torch.zeros(size, dtype=torch.uint8, device=DEV)
    score = torch.full((n,), -1.0, device=DEV)
    mask = torch.full((n,), 7, dtype=torch.uint8, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.tee_exit_gate(ctypes.byref(desc), n, p(h), h.stride(0), None, 0, None, p(w["w_down"]), None,
                           p(w["w_up"]), None, p(score), p(mask), None, p(ws), size, stream)
    assert st == _lib.TEE_OK
    torch.cuda.synchronize()
    p_ref, _, _ = _router_ref(h, w, 0.5, "per_token", eps=cfg.eps)
    check_scores(score, p_ref)
    check_mask(mask, p_ref, 0.5)
    assert int(ws[:8].view(torch.int32)[0].item()) == 0


def test_router_calls_share_a_workspace(tee):
    # tensor-core and CUDA-core calls alternate on one workspace: each must see clean sums
    cfg = configs.ROUTER_4096
    ws = tee.Workspace(DEV)
    w = gen.router_weights(cfg, 11, seed=1, device=DEV)
    for n in (4096, 64, 20000, 4096, 300, 20000, 300):
        h = gen.router_hidden(cfg, n, 11, seed=n, device=DEV)
        score, mask, _ = tee.exit_gate(h, 0.5, w_down=w["w_down"], w_up=w["w_up"], eps=cfg.eps, ws=ws)
        p_ref, _, _ = _router_ref(h, w, 0.5, "per_token", eps=cfg.eps)
        check_scores(score, p_ref)
    assert ws.device_error() == (0, 0)
