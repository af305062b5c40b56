"""Pins of the oracle's KV fill, int4 dequantisation, RoPE and ridge fit (no GPU)."""
import cmath
import math

import numpy as np
import pytest

import oracle
from oracle.fill import layer_weights
from workloads import configs, gen

RNG = np.random.default_rng(99)
S2 = math.sqrt(2.0)


# ------------------------------------------------------------------ int4

def test_dequant_worked_example():
    # byte 0x1F holds q=15 (even k, low nibble) and q=1 (odd k, high nibble).
    packed = np.array([[0x1F], [0x80]], dtype=np.uint8)          # k = 0..3, one column
    scale = np.array([[0.5], [0.25]])                              # group = 2 rows
    zero = np.array([[7.5], [8.0]])
    w = oracle.dequant_int4(packed, scale, zero, group=2)
    np.testing.assert_array_equal(w[:, 0], [(15 - 7.5) * 0.5, (1 - 7.5) * 0.5,
                                            (0 - 8.0) * 0.25, (8 - 8.0) * 0.25])


def test_dequant_round_trips_exactly_representable_weights():
    d, kvw, g = 128, 8, 64
    q = RNG.integers(0, 16, (d, kvw))
    s = RNG.choice([0.5, 0.25, 0.125], (d // g, kvw))
    z = RNG.choice([7.5, 8.0, 6.75], (d // g, kvw))
    dense = (q - np.repeat(z, g, 0)) * np.repeat(s, g, 0)
    import torch
    packed = gen.pack_int4(torch.from_numpy(q.astype(np.uint8))).numpy()
    np.testing.assert_array_equal(oracle.dequant_int4(packed, s, z, g), dense)


# ------------------------------------------------------------------ RoPE

def test_rope_position_zero_is_identity():
    k = RNG.standard_normal((3, 2, 64))
    np.testing.assert_array_equal(oracle.rope_rotate_half(k, np.zeros((3, 1)), 1e4), k)


def test_rope_is_complex_multiplication_of_half_pairs():
    # Element i and i + hd/2 form z_i = k_i + 1j k_{i+hd/2}; RoPE multiplies z_i
    # by exp(1j * pos * base^(-2i/hd)).
    hd, base = 8, 10000.0
    k = RNG.standard_normal(hd)
    for pos in (1, 7, 123457):
        got = oracle.rope_rotate_half(k, np.array(pos), base)
        for i in range(hd // 2):
            z = complex(k[i], k[i + hd // 2]) * cmath.exp(1j * pos * base ** (-2 * i / hd))
            assert abs(got[i] - z.real) < 1e-9 and abs(got[i + hd // 2] - z.imag) < 1e-9


def test_rope_quarter_turn_closed_form():
    # hd = 4: pair (1, 3) turns by pos * base^(-1/2). base = (2*pos/pi)^2 makes
    # that exactly pi/2, so (k1, k3) -> (-k3, k1).
    pos = 3
    base = (2 * pos / math.pi) ** 2
    got = oracle.rope_rotate_half(np.array([0.0, 1.0, 0.0, 2.0]), np.array(pos), base)
    np.testing.assert_allclose(got, [0.0, -2.0, 0.0, 1.0], atol=1e-15)


def test_rope_keeps_pair_norms_and_depends_on_relative_position():
    hd = 64
    q, k = RNG.standard_normal(hd), RNG.standard_normal(hd)
    rq = oracle.rope_rotate_half(q, np.array(1000), 5e5)
    pn = lambda v: v[: hd // 2] ** 2 + v[hd // 2:] ** 2  # noqa: E731
    np.testing.assert_allclose(pn(rq), pn(q), rtol=1e-12)
    dots = [oracle.rope_rotate_half(q, np.array(m), 5e5) @ oracle.rope_rotate_half(k, np.array(m - 17), 5e5)
            for m in (17, 100, 5000)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ------------------------------------------------------------------ fill

def _layer(d, kvw, w_map=None, gamma=None, wk=None, wv=None, cache_layer=0):
    return {"w_map": w_map, "gamma": np.ones(d) if gamma is None else gamma,
            "wk": RNG.standard_normal((d, kvw)) if wk is None else wk,
            "wv": RNG.standard_normal((d, kvw)) if wv is None else wv, "cache_layer": cache_layer}


def test_fill_worked_example_identity_map():
    # h = (3, 4): RMSNorm -> (3 sqrt2/5, 4 sqrt2/5); Wk = I, Wv swaps the two
    # columns; one head of width 2 at position 0 (no rotation).
    L = _layer(2, 2, wk=np.eye(2), wv=np.array([[0.0, 1.0], [1.0, 0.0]]))
    k, v = oracle.fill_rows(np.array([[3.0, 4.0]]), L, [0], 1, 2, 1e4, eps=0.0)
    np.testing.assert_allclose(k[0, 0], [3 * S2 / 5, 4 * S2 / 5], atol=1e-15)
    np.testing.assert_allclose(v[0, 0], [4 * S2 / 5, 3 * S2 / 5], atol=1e-15)


def test_fill_map_is_a_row_vector_times_w():
    # x = h W with W = [[1, 1], [0, 1]] gives (3, 7) from h = (3, 4) (W h would
    # give (7, 4)); RMSNorm -> (3, 7)/sqrt(29).
    L = _layer(2, 2, w_map=np.array([[1.0, 1.0], [0.0, 1.0]]), wk=np.eye(2), wv=np.eye(2))
    k, v = oracle.fill_rows(np.array([[3.0, 4.0]]), L, [0], 1, 2, 1e4, eps=0.0)
    np.testing.assert_allclose(k[0, 0], [3 / math.sqrt(29), 7 / math.sqrt(29)], atol=1e-15)


def test_fill_with_identity_reproduces_backbone_kv_on_exact_inputs():
    # Backbone K/V of a layer whose exact input is x, computed head by head with
    # complex rotations; a fill whose map turns h into x exactly (a permutation)
    # must write the same K/V.
    d, nkv, hd, base, eps = 16, 2, 4, 1e4, 1e-5
    perm = RNG.permutation(d)
    P = np.eye(d)[:, perm]                    # (h P)[n] = h[perm[n]]
    h = RNG.standard_normal((3, d))
    x = h[:, perm]
    g = 1 + 0.1 * RNG.standard_normal(d)
    wk, wv = RNG.standard_normal((d, nkv * hd)), RNG.standard_normal((d, nkv * hd))
    pos = [0, 5, 77]
    for w_map, inp in ((None, x), (P, h)):
        k, v = oracle.fill_rows(inp, _layer(d, nkv * hd, w_map, g, wk, wv), pos, nkv, hd, base, eps)
        for t in range(3):
            xn = x[t] / (np.linalg.norm(x[t]) / math.sqrt(d)) if eps == 0 else \
                x[t] / math.sqrt(np.dot(x[t], x[t]) / d + eps)
            kk, vv = (xn * g) @ wk, (xn * g) @ wv
            for hh in range(nkv):
                np.testing.assert_allclose(v[t, hh], vv[hh * hd:(hh + 1) * hd], rtol=1e-12)
                for i in range(hd // 2):
                    z = complex(kk[hh * hd + i], kk[hh * hd + i + hd // 2]) * \
                        cmath.exp(1j * pos[t] * base ** (-2 * i / hd))
                    assert abs(k[t, hh, i] - z.real) < 1e-10
                    assert abs(k[t, hh, i + hd // 2] - z.imag) < 1e-10


def test_fill_is_scale_invariant_and_linear_in_gamma():
    d, kvw = 32, 8
    h = RNG.standard_normal((4, d))
    L = _layer(d, kvw, w_map=RNG.standard_normal((d, d)) / math.sqrt(d))
    k1, v1 = oracle.fill_rows(h, L, [1, 2, 3, 4], 2, 4, 1e4, eps=0.0)
    k2, v2 = oracle.fill_rows(6.0 * h, L, [1, 2, 3, 4], 2, 4, 1e4, eps=0.0)
    np.testing.assert_allclose(k1, k2, rtol=1e-12)
    L2 = dict(L, gamma=2.5 * np.ones(d))
    k3, v3 = oracle.fill_rows(h, L2, [1, 2, 3, 4], 2, 4, 1e4, eps=0.0)
    np.testing.assert_allclose(k3, 2.5 * k1, rtol=1e-12)
    np.testing.assert_allclose(v3, 2.5 * v1, rtol=1e-12)


def test_w4a16_fill_equals_dense_fill_on_dequantised_weights():
    cfg = configs.DecodeConfig(**{**configs.LLAMA1B_DECODE.__dict__, "d": 128, "batch": 4})
    x = gen.decode_inputs(cfg, seed=1, device="cpu", case="exit", with_cache=False)
    L = {k: (v.float().numpy() if hasattr(v, "float") and v.dtype.is_floating_point else
             (v.numpy() if hasattr(v, "numpy") else v)) for k, v in x["layers"][0].items()}
    wk, wv = layer_weights(L)
    dense = {"w_map": None, "gamma": L["gamma"], "wk": wk, "wv": wv, "cache_layer": 0}
    h = x["h_cur"].float().numpy()
    a = oracle.fill_rows(h, L, [0, 1, 2, 3], cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps)
    b = oracle.fill_rows(h, dense, [0, 1, 2, 3], cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_kv_fill_writes_exactly_the_backbone_slots():
    d, nkv, hd = 8, 2, 4
    sent = -7.0
    kc = np.full((2, 3, nkv, 5, hd), sent)
    vc = np.full((2, 3, nkv, 5, hd), sent)
    h = RNG.standard_normal((4, d))
    L = _layer(d, nkv * hd, cache_layer=1)
    # fill local rows 3 and 1: row 3 is sequence 2 at position 4, row 1 is sequence 0 at position 2
    pos = np.array([0, 2, 0, 4])
    seq = np.array([0, 0, 1, 2])
    k2, v2 = oracle.kv_fill(h, [L], kc, vc, nkv, hd, 1e4, 1e-5, rows=[3, 1], pos=pos, seq=seq)
    k_ref, v_ref = oracle.fill_rows(h[[3, 1]], L, [4, 2], nkv, hd, 1e4, 1e-5)
    np.testing.assert_array_equal(k2[1, 2, :, 4], k_ref[0])
    np.testing.assert_array_equal(v2[1, 0, :, 2], v_ref[1])
    written = np.zeros(kc.shape, bool)
    written[1, 2, :, 4] = True
    written[1, 0, :, 2] = True
    assert np.all(k2[~written] == sent) and np.all(v2[~written] == sent)
    # default addressing: row r -> position pos0 + r of sequence 0
    k3, _ = oracle.kv_fill(h[:2], [L], kc, vc, nkv, hd, 1e4, 1e-5, pos0=3)
    k_ref, _ = oracle.fill_rows(h[:2], L, [3, 4], nkv, hd, 1e4, 1e-5)
    np.testing.assert_array_equal(k3[1, 0, :, 3], k_ref[0])
    np.testing.assert_array_equal(k3[1, 0, :, 4], k_ref[1])


# ------------------------------------------------------------------ model-family variants

def test_fill_bias_with_zero_weights_is_the_bias():
    # Wk = Wv = 0: k = k_bias, v = v_bias; at position 0 RoPE leaves k as it is
    d, nkv, hd = 4, 2, 2
    kb, vb = np.array([1.0, -2.0, 0.5, 3.0]), np.array([-1.0, 0.25, 2.0, 7.0])
    L = _layer(d, nkv * hd, wk=np.zeros((d, nkv * hd)), wv=np.zeros((d, nkv * hd)))
    L["k_bias"], L["v_bias"] = kb, vb
    k, v = oracle.fill_rows(RNG.standard_normal((1, d)), L, [0], nkv, hd, 1e4, 1e-5)
    np.testing.assert_array_equal(k[0].ravel(), kb)
    np.testing.assert_array_equal(v[0].ravel(), vb)
    # at position p the bias is rotated like any k: head (1, -2) by angle p (i = 0, hd = 2)
    k, _ = oracle.fill_rows(RNG.standard_normal((1, d)), L, [1], nkv, hd, 1e4, 1e-5)
    c, sn = math.cos(1.0), math.sin(1.0)
    np.testing.assert_allclose(k[0, 0], [1.0 * c + 2.0 * sn, -2.0 * c + 1.0 * sn], atol=1e-15)


def test_qk_norm_normalises_each_head_before_rope():
    # worked example: one head k = (3, 4) at position 0, k_norm = (1, 1), eps = 0:
    # mean square 12.5, k -> (3, 4)/sqrt(12.5)
    d = 2
    L = _layer(d, 2, wk=np.eye(2), wv=np.eye(2))
    L["k_norm"] = np.ones(2)
    h = np.array([[3.0, 4.0]])
    k, v = oracle.fill_rows(h, L, [0], 1, 2, 1e4, eps=0.0)
    xn = h / math.sqrt(12.5)   # the layer norm already gives unit mean square
    np.testing.assert_allclose(k[0, 0], xn[0], atol=1e-15)
    np.testing.assert_allclose(v[0, 0], xn[0], atol=1e-15)   # v is not normalised by k_norm
    # any head: mean square 1 before RoPE (which keeps pair norms, so also after), scaled by k_norm
    d, nkv, hd = 16, 2, 8
    L = _layer(d, nkv * hd)
    L["k_bias"] = RNG.standard_normal(nkv * hd)
    L["k_norm"] = np.full(hd, 2.0)
    k, _ = oracle.fill_rows(RNG.standard_normal((3, d)), L, [0, 5, 9], nkv, hd, 1e4, eps=0.0)
    np.testing.assert_allclose(np.mean(k * k, axis=-1), 4.0, rtol=1e-12)


def test_k_only_and_v_only_fills_keep_the_other_cache():
    d, nkv, hd = 8, 2, 4
    kc = np.full((1, 1, nkv, 4, hd), -3.0)
    vc = np.full((1, 1, nkv, 4, hd), -5.0)
    h = RNG.standard_normal((2, d))
    for w, k_written, v_written in (("k", True, False), ("v", False, True), (1, True, False), (2, False, True),
                                    (None, True, True)):
        L = _layer(d, nkv * hd, cache_layer=0)
        L["writes"] = w
        k2, v2 = oracle.kv_fill(h, [L], kc, vc, nkv, hd, 1e4, 1e-5)
        assert bool(np.any(k2 != -3.0)) == k_written
        assert bool(np.any(v2 != -5.0)) == v_written


# ------------------------------------------------------------------ ridge

def test_ridge_with_orthonormal_columns():
    X, _ = np.linalg.qr(RNG.standard_normal((40, 6)))
    Y = RNG.standard_normal((40, 3))
    np.testing.assert_allclose(oracle.ridge_fit(X, Y, 0.3), X.T @ Y / 1.3, atol=1e-13)


def test_ridge_recovers_a_as_lambda_goes_to_zero():
    X = RNG.standard_normal((50, 5))
    A = RNG.standard_normal((5, 4))
    errs = [np.abs(oracle.ridge_fit(X, X @ A, lam) - A).max() for lam in (1e-2, 1e-4, 1e-6)]
    assert errs[0] < 1e-2 and errs[2] < 1e-6
    assert 50 < errs[0] / errs[1] < 200 and 50 < errs[1] / errs[2] < 200  # error O(lambda)


def test_ridge_equals_augmented_least_squares():
    X = RNG.standard_normal((30, 7))
    Y = RNG.standard_normal((30, 2))
    lam = 0.7
    Xa = np.vstack([X, math.sqrt(lam) * np.eye(7)])
    Ya = np.vstack([Y, np.zeros((7, 2))])
    np.testing.assert_allclose(oracle.ridge_fit(X, Y, lam), np.linalg.lstsq(Xa, Ya, rcond=None)[0], atol=1e-12)
