"""Pins of the oracle's exit gates against closed forms, invariants, worked
examples and the pages' printed numbers (no GPU)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from workloads import configs, gen

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- cosine gate

def test_cosine_of_itself_and_scaled_copies():
    x = RNG.standard_normal((5, 37))
    np.testing.assert_allclose(oracle.cosine_similarity(x, x), 1.0, atol=1e-15)
    np.testing.assert_allclose(oracle.cosine_similarity(x, 3.5 * x), 1.0, atol=1e-15)
    np.testing.assert_allclose(oracle.cosine_similarity(x, -0.25 * x), -1.0, atol=1e-15)


def test_cosine_of_orthogonal_basis_vectors_is_zero():
    e = np.eye(6)
    s = oracle.cosine_similarity(e[[0, 1, 2]], e[[3, 5, 4]])
    assert np.all(s == 0.0)


def test_cosine_worked_examples():
    # (1,2,2).(2,1,2) = 8, both norms 3  ->  8/9
    # (1,0,0,0).(1,1,1,1) = 1, norms 1 and 2  ->  1/2
    # (1,1).(1,-1) = 0
    a = np.array([[1, 2, 2, 0], [1, 0, 0, 0], [1, 1, 0, 0]], dtype=float)
    b = np.array([[2, 1, 2, 0], [1, 1, 1, 1], [1, -1, 0, 0]], dtype=float)
    np.testing.assert_allclose(oracle.cosine_similarity(a, b), [8 / 9, 0.5, 0.0], atol=1e-15)


def test_cosine_scale_invariance_and_chord_identity():
    a = RNG.standard_normal((9, 64))
    b = RNG.standard_normal((9, 64))
    s = oracle.cosine_similarity(a, b)
    np.testing.assert_allclose(oracle.cosine_similarity(2.0 * a, 0.125 * b), s, atol=1e-14)
    # For unit vectors, cos = 1 - |u - v|^2 / 2 (law of cosines).
    u = a / np.linalg.norm(a, axis=1, keepdims=True)
    v = b / np.linalg.norm(b, axis=1, keepdims=True)
    np.testing.assert_allclose(s, 1.0 - np.sum((u - v) ** 2, axis=1) / 2.0, atol=1e-14)


def test_cosine_zero_row_never_exits():
    a = np.zeros((1, 8))
    b = np.ones((1, 8))
    s, mask, flag = oracle.cosine_gate(a, b, tau=-0.5)
    assert s[0] == 0.0 and mask[0] == 1  # 0 > -0.5 is an exit for a negative tau
    s, mask, flag = oracle.cosine_gate(a, b, tau=0.0)
    assert mask[0] == 0 and flag == 0


def test_exit_is_strict_at_the_threshold():
    # A token whose similarity equals tau exactly does not exit (strict ">").
    a = np.array([[1.0, 0.0]])
    b = np.array([[1.0, 0.0]])
    _, mask, _ = oracle.cosine_gate(a, b, tau=1.0)
    assert mask[0] == 0
    _, mask, _ = oracle.cosine_gate(a, b, tau=np.nextafter(np.float32(1.0), np.float32(0.0)))
    assert mask[0] == 1


def test_batch_min_rule():
    # Four tokens with similarities (cos 0, cos 0.1, cos 0.2, cos 0.3) rad apart.
    ang = np.array([0.0, 0.1, 0.2, 0.3])
    a = np.stack([np.ones_like(ang), np.zeros_like(ang)], axis=1)
    b = np.stack([np.cos(ang), np.sin(ang)], axis=1)
    tau = 0.97  # cos(0.2) = 0.980, cos(0.3) = 0.955
    s, m_tok, f_tok = oracle.cosine_gate(a, b, tau, "per_token")
    np.testing.assert_allclose(s, np.cos(ang), atol=1e-15)
    assert list(m_tok) == [1, 1, 1, 0] and f_tok == 0
    s, m_all, f_all = oracle.cosine_gate(a, b, tau, "batch_all")
    assert list(m_all) == [0, 0, 0, 0] and f_all == 0
    s, m_all, f_all = oracle.cosine_gate(a[:3], b[:3], tau, "batch_all")
    assert list(m_all) == [1, 1, 1] and f_all == 1


def test_beta81_exit_fraction_matches_closed_form():
    # a ~ Beta(8,1) has CDF a^8, so P(a > tau) = 1 - tau^8; for large d the
    # cosine of the generator's pair concentrates at a.
    cfg = configs.DecodeConfig(**{**configs.TINY_DECODE.__dict__, "batch": 6000, "d": 4096})
    x = gen.decode_inputs(cfg, seed=3, device="cpu", with_cache=False)
    s, mask, _ = oracle.cosine_gate(x["h_prev"].double().numpy(), x["h_cur"].double().numpy(), 0.95)
    expect = 1.0 - 0.95 ** 8
    assert abs(mask.mean() - expect) < 0.02, (mask.mean(), expect)
    assert np.abs(s - x["a"].double().numpy()).max() < 0.06


def test_bf16_batch_min_cases_of_the_decode_workload():
    cfg = configs.LLAMA1B_DECODE
    for case, want in (("exit", 1), ("stay", 0)):
        x = gen.decode_inputs(cfg, seed=0, device="cpu", case=case, with_cache=False)
        _, mask, flag = oracle.cosine_gate(x["h_prev"].float().numpy(), x["h_cur"].float().numpy(),
                                           cfg.tau, "batch_all")
        assert flag == want and int(mask.sum()) == want * cfg.batch


# ---------------------------------------------------------------- router gate

LN3 = math.log(3.0)


def test_router_zero_weights_give_sigmoid_of_bias():
    h = RNG.standard_normal((7, 32))
    wd, wu = np.zeros((128, 32)), np.zeros(128)
    assert np.all(oracle.router_probability(h, wd, wu) == 0.5)
    p = oracle.router_probability(h, wd, wu, b_up=np.array([LN3]))
    np.testing.assert_allclose(p, 0.75, atol=1e-15)  # sigmoid(ln 3) = 3/4


def test_router_closed_form_silu_and_bias_placement():
    # W_down = 0 and b_down = ln 3 make u = ln 3 on every channel;
    # SiLU(ln 3) = ln 3 * 3/4. With W_up = 1 on one channel and
    # b_up = ln(3)/4, z = 3/4 ln 3 + 1/4 ln 3 = ln 3 and p = 3/4.
    h = RNG.standard_normal((3, 16))
    p = oracle.router_probability(h, np.zeros((1, 16)), np.array([1.0]),
                                  b_down=np.array([LN3]), b_up=np.array([LN3 / 4]))
    np.testing.assert_allclose(p, 0.75, atol=1e-15)
    # Two channels each carrying half of W_up sum to the same z.
    p = oracle.router_probability(h, np.zeros((2, 16)), np.array([0.5, 0.5]),
                                  b_down=np.array([LN3, LN3]), b_up=np.array([LN3 / 4]))
    np.testing.assert_allclose(p, 0.75, atol=1e-15)


def test_router_closed_form_rmsnorm_mean_not_sum():
    # h = (ln 3, sqrt(2 - ln^2 3)) has mean(h^2) = 1, so RMSNorm leaves it
    # unchanged (eps = 0) and W_down = (1, 0) gives u = ln 3 -> p = 3/4.
    # Scaling h by 5 must not change p (RMSNorm is scale-invariant).
    h = np.array([[LN3, math.sqrt(2 - LN3 ** 2)]])
    kw = dict(b_up=np.array([LN3 / 4]), eps=0.0)
    np.testing.assert_allclose(oracle.router_probability(h, np.array([[1.0, 0.0]]), np.array([1.0]), **kw), 0.75, atol=1e-15)
    np.testing.assert_allclose(oracle.router_probability(5 * h, np.array([[1.0, 0.0]]), np.array([1.0]), **kw), 0.75, atol=1e-15)
    # gamma scales the normalised vector, not the input of the norm:
    # gamma = (2, 7) with W_down = (0.5, 0) gives the same u.
    np.testing.assert_allclose(
        oracle.router_probability(h, np.array([[0.5, 0.0]]), np.array([1.0]), gamma=np.array([2.0, 7.0]), **kw),
        0.75, atol=1e-15)


def test_router_gamma_folds_into_w_down_and_is_scale_invariant():
    h = RNG.standard_normal((6, 48))
    wd = 0.02 * RNG.standard_normal((128, 48))
    wu = 0.02 * RNG.standard_normal(128)
    g = 1 + 0.1 * RNG.standard_normal(48)
    p1 = oracle.router_probability(h, wd, wu, gamma=g)
    p2 = oracle.router_probability(h, wd * g[None, :], wu)
    np.testing.assert_allclose(p1, p2, atol=1e-15)
    np.testing.assert_allclose(oracle.router_probability(9.0 * h, wd, wu, eps=0.0),
                               oracle.router_probability(h, wd, wu, eps=0.0), atol=1e-14)
    # W_up = 0: p does not depend on h.
    p = oracle.router_probability(h, wd, np.zeros(128), b_up=np.array([0.3]))
    np.testing.assert_allclose(p, 1 / (1 + math.exp(-0.3)), atol=1e-15)


def test_router_shapes_match_the_printed_parameter_count(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tide_router_params.json")))
    d, b = g["d"], g["bottleneck"]
    wd, wu = np.zeros((b, d)), np.zeros(b)
    assert wd.size + wu.size == g["params_exact"]
    assert abs(g["params_exact"] - g["params_printed_approx"]) < 1000
    h = np.ones((1, d))
    oracle.router_probability(h, wd, wu)
    with pytest.raises(ValueError):
        oracle.router_probability(h, wd.T, wu)  # W_down must be b x d


def test_router_distribution_of_the_workload():
    # Weights N(0, 0.02^2), gamma 1: p stays near 1/2 (spread ~0.05), so
    # about half the tokens exit at theta = 0.5 and almost none at 0.9.
    cfg = configs.ROUTER_4096
    w = gen.router_weights(cfg, cfg.checkpoints[0], seed=0)
    h = gen.router_hidden(cfg, 512, cfg.checkpoints[0], seed=0)
    p = oracle.router_probability(h.float().numpy(), w["w_down"].float().numpy(), w["w_up"].float().numpy())
    assert 0.3 < (p > 0.5).mean() < 0.7
    assert (p > 0.9).mean() == 0.0
    assert 0.01 < p.std() < 0.2


# ------------------------------------------------------- cascade accounting

def test_tide_figure2_layer_ops(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tide_fig2_layer_ops.json")))
    L = g["n_layers"]
    ckpts = [k for k in range(L) if (k + 1) % 4 == 0]
    # 'the' passes first at the checkpoint after layer 8, 'cat' after 16, 'sat' never.
    probs = {k: np.array([0.9 if k >= 7 else 0.1, 0.9 if k >= 15 else 0.2, 0.3]) for k in ckpts}
    depth = oracle.earliest_exit(probs, theta=0.5, n_layers=L)
    assert list(depth) == g["exit_depth"]
    ops = oracle.layer_ops(depth)
    assert ops == g["layer_ops"] and len(depth) * L == g["baseline_ops"]
    assert round(100 * (1 - ops / g["baseline_ops"])) == g["reduction_percent_printed"]
    # k_min = 8 skips checkpoint 7, so 'the' exits at the next one (layer 11, depth 12).
    depth = oracle.earliest_exit(probs, theta=0.5, n_layers=L, k_min=8)
    assert list(depth) == [12, 16, 32]


def test_checkpoint_set_matches_printed_layers(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tide_calibration_config.json")))
    for m in g["models"]:
        ck = [k for k in range(m["n_layers"]) if (k + 1) % g["interval"] == 0]
        assert m["printed_layer"] in ck
    assert configs.ROUTER_4096.checkpoints == tuple(range(3, 32, 4))
