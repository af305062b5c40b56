"""Pins of the Exit River oracle against closed forms, a library routine and the
fill oracle (which is pinned on its own)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import river
from tests.parity import host
from workloads import configs, gen

RNG = np.random.default_rng(2024)


def _tiny(seed=0):
    cfg = configs.TINY_RIVER
    x = host(gen.river_inputs(cfg, seed))
    return cfg, x


def _run(cfg, x, layers=None):
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    out = river.exit_river(x["h"], x["layers"] if layers is None else layers, x["pos"], x["seq"], kc, vc,
                           cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    return out, kc, vc


def _zero(L, m):
    L[f"{m}_scale"] = np.zeros_like(L[f"{m}_scale"])


def test_silu_closed_forms():
    a = np.array([0.0, 2.0, -2.0, 40.0, -40.0])
    s = river.silu(a)
    assert s[0] == 0.0
    assert abs(s[1] - 2.0 / (1.0 + math.exp(-2.0))) < 1e-15 and abs(s[1] - 1.7615941559557649) < 1e-15
    assert abs(s[3] - 40.0) < 1e-12 and abs(s[4]) < 1e-15
    x = RNG.standard_normal(100) * 5
    np.testing.assert_allclose(river.silu(x) - river.silu(-x), x, atol=1e-12)   # sigma(x) + sigma(-x) = 1


@pytest.mark.parametrize("n_q,n_kv", [(4, 2), (8, 8), (6, 1)])
def test_attention_is_the_library_causal_attention(n_q, n_kv):
    # each item: softmax(q k^T / sqrt(hd)) v over positions 0..pos, q head h on kv head h // (n_q / n_kv)
    n, hd, P, S = 5, 16, 12, 3
    q = RNG.standard_normal((n, n_q, hd))
    kc = RNG.standard_normal((S, n_kv, P, hd))
    vc = RNG.standard_normal((S, n_kv, P, hd))
    pos = np.array([0, 11, 5, 7, 3])
    seq = np.array([0, 2, 1, 2, 0])
    o = river.attention(q, kc, vc, pos, seq, n_kv)
    rep = n_q // n_kv
    for i in range(n):
        p, s = pos[i], seq[i]
        k = torch.from_numpy(kc[s, :, :p + 1]).repeat_interleave(rep, dim=0)[None]
        v = torch.from_numpy(vc[s, :, :p + 1]).repeat_interleave(rep, dim=0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q[i])[None, :, None, :], k, v)
        np.testing.assert_allclose(o[i], ref[0, :, 0].numpy(), atol=1e-12)


def test_attention_with_equal_keys_averages_the_values():
    n_q, n_kv, hd, P = 4, 2, 8, 9
    kc = np.zeros((1, n_kv, P, hd))
    vc = RNG.standard_normal((1, n_kv, P, hd))
    q = RNG.standard_normal((2, n_q, hd))
    o = river.attention(q, kc, vc, np.array([8, 3]), np.array([0, 0]), n_kv)
    for h in range(n_q):
        np.testing.assert_allclose(o[0, h], vc[0, h // 2, :9].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(o[1, h], vc[0, h // 2, :4].mean(axis=0), atol=1e-14)


def test_zero_output_projections_keep_h_and_write_the_fill_kv():
    # Wo = Wd = 0: the hidden state passes unchanged, and the cache slots hold
    # what the (separately pinned) fill oracle writes for the same Wk, Wv, norm
    cfg, x = _tiny(1)
    for L in x["layers"]:
        _zero(L, "o")
        _zero(L, "d")
    out, kc, vc = _run(cfg, x)
    np.testing.assert_array_equal(out, x["h"])
    for L in x["layers"]:
        fl = {"cache_layer": L["cache_layer"], "w_map": None, "gamma": L["attn_norm"], "wk": L["wk"],
              "wv": L["wv"], "k_scale": L["k_scale"], "k_zero": L["k_zero"], "v_scale": L["v_scale"],
              "v_zero": L["v_zero"]}
        k_ref, v_ref = oracle.fill_rows(x["h"], fl, x["pos"], cfg.n_kv_heads, cfg.head_dim, cfg.rope_base,
                                        cfg.eps, cfg.group)
        j = L["cache_layer"]
        np.testing.assert_allclose(kc[j, x["seq"], :, x["pos"]], k_ref, atol=1e-12)
        np.testing.assert_allclose(vc[j, x["seq"], :, x["pos"]], v_ref, atol=1e-12)
    # nothing else moved
    mask = np.ones(kc.shape[:4], dtype=bool)
    for L in x["layers"]:
        mask[L["cache_layer"], x["seq"], :, x["pos"]] = False
    np.testing.assert_array_equal(kc[mask], x["k_cache"][mask])
    np.testing.assert_array_equal(vc[mask], x["v_cache"][mask])


def test_zero_gate_switches_the_ffn_off():
    # Wg = 0: SiLU(0) = 0 gates every hidden unit, so h' = h1 = h + o Wo
    cfg, x = _tiny(2)
    L = x["layers"][0]
    _zero(L, "g")
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    out = river.exit_layer(x["h"], L, x["pos"], x["seq"], kc, vc, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                           cfg.rope_base, cfg.eps, cfg.group)
    _zero(L, "d")
    kc2, vc2 = x["k_cache"].copy(), x["v_cache"].copy()
    out2 = river.exit_layer(x["h"], L, x["pos"], x["seq"], kc2, vc2, cfg.n_q_heads, cfg.n_kv_heads,
                            cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    np.testing.assert_array_equal(out, out2)
    assert np.abs(out - x["h"]).max() > 0.01   # the attention half still acts


def test_first_position_attends_to_its_own_value():
    # pos = 0: the softmax has one term, so every q head's output is the token's
    # own V of its kv head, i.e. h1 = h + [v_(h // rep)]_h Wo; with Wd = 0, h' = h1
    cfg, x = _tiny(3)
    x["pos"] = np.zeros_like(x["pos"])
    L = x["layers"][0]
    _zero(L, "d")
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    out = river.exit_layer(x["h"], L, x["pos"], x["seq"], kc, vc, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                           cfg.rope_base, cfg.eps, cfg.group)
    v = vc[L["cache_layer"], x["seq"], :, 0]                     # [n][n_kv][hd], just written
    rep = cfg.n_q_heads // cfg.n_kv_heads
    o = np.repeat(v, rep, axis=1).reshape(len(x["h"]), -1)
    np.testing.assert_allclose(out, x["h"] + o @ river.weight(L, "o", cfg.group), atol=1e-12)


def _w4(dense, scale):
    # exactly representable int4 weights: codes dense / scale + 8, zero 8, group 2
    codes = (np.asarray(dense) / scale + 8).astype(np.uint8)
    packed = codes[0::2] | (codes[1::2] << 4)
    k, n = codes.shape
    return packed, np.full((k // 2, n), scale), np.full((k // 2, n), 8.0)


def test_ffn_reads_the_attention_residual_worked_example():
    # d = 4, one head of width 2, position 0 (o = the token's own v), unit norm
    # weights, eps = 0. h = (2, 0, 0, 0) -> x = h; v = x Wv = (2, 0); o = v;
    # h1 = h + o Wo = (2, 2, 0, 0); x2 = h1 / rms(h1) = (sqrt2, sqrt2, 0, 0);
    # gate = 2 sqrt2, up = sqrt2, a = SiLU(2 sqrt2) sqrt2 = 4 / (1 + e^(-2 sqrt2));
    # out = h1 + a (1, 0, 0, 0)
    L = {"cache_layer": 0, "attn_norm": np.ones(4), "ffn_norm": np.ones(4)}
    z42 = np.zeros((4, 2))
    for m, dense, s in (("q", z42, 1.0), ("k", z42, 1.0), ("v", [[1.0, 0], [0, 0], [0, 0], [0, 0]], 1.0),
                        ("o", [[0, 1.0, 0, 0], [0, 0, 0, 0]], 1.0), ("g", [[1.0, 0], [1.0, 0], [0, 0], [0, 0]], 1.0),
                        ("u", [[0.5, 0], [0.5, 0], [0, 0], [0, 0]], 0.5), ("d", [[1.0, 0, 0, 0], [0, 0, 0, 0]], 1.0)):
        L[f"w{m}"], L[f"{m}_scale"], L[f"{m}_zero"] = _w4(dense, s)
    kc = np.zeros((1, 1, 1, 4, 2))
    vc = np.zeros((1, 1, 1, 4, 2))
    out = river.exit_layer(np.array([[2.0, 0, 0, 0]]), L, [0], [0], kc, vc, 1, 1, 2, 1e4, 0.0, group=2)
    a = 4.0 / (1.0 + math.exp(-2.0 * math.sqrt(2.0)))
    np.testing.assert_allclose(out, [[2.0 + a, 2.0, 0, 0]], atol=1e-14)


def test_one_hidden_unit_worked_example():
    # d = 4, one q/kv head of width 2 with Wo = 0; FFN of one hidden unit with
    # exactly representable int4 weights (group 2): h = (2, 0, 0, 0), unit norm
    # weights, eps = 0 -> x2 = (2, 0, 0, 0); gate = 1 * 2, up = 0.5 * 2 = 1,
    # a = SiLU(2) * 1 = 2 / (1 + e^-2); out = h + a * (1, 0, 0, 0)
    def w4(dense, scale):
        codes = (np.asarray(dense) / scale + 8).astype(np.uint8)   # z = 8
        packed = codes[0::2] | (codes[1::2] << 4)
        k, n = codes.shape
        return packed, np.full((k // 2, n), scale), np.full((k // 2, n), 8.0)

    L = {"cache_layer": 0, "attn_norm": np.ones(4), "ffn_norm": np.ones(4)}
    for m, dense, s in (("q", np.zeros((4, 2)), 1.0), ("k", np.zeros((4, 2)), 1.0), ("v", np.zeros((4, 2)), 1.0),
                        ("o", np.zeros((2, 4)), 1.0), ("g", [[1.0, 0.0], [0, 0], [0, 0], [0, 0]], 1.0),
                        ("u", [[0.5, 0.0], [0, 0], [0, 0], [0, 0]], 0.5),
                        ("d", [[1.0, 0, 0, 0], [0, 0, 0, 0]], 1.0)):
        L[f"w{m}"], L[f"{m}_scale"], L[f"{m}_zero"] = w4(dense, s)
    kc = np.zeros((1, 1, 1, 4, 2))
    vc = np.zeros((1, 1, 1, 4, 2))
    out = river.exit_layer(np.array([[2.0, 0, 0, 0]]), L, [3], [0], kc, vc, 1, 1, 2, 1e4, 0.0, group=2)
    np.testing.assert_allclose(out, [[2.0 + 1.7615941559557649, 0, 0, 0]], atol=1e-15)


def test_river_is_the_layers_in_order():
    cfg, x = _tiny(4)
    out, kc, vc = _run(cfg, x)
    kc2, vc2 = x["k_cache"].copy(), x["v_cache"].copy()
    hmid = river.exit_layer(x["h"], x["layers"][0], x["pos"], x["seq"], kc2, vc2, cfg.n_q_heads, cfg.n_kv_heads,
                            cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    out2 = river.exit_layer(hmid, x["layers"][1], x["pos"], x["seq"], kc2, vc2, cfg.n_q_heads, cfg.n_kv_heads,
                            cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(kc, kc2)
    # the second layer reads the first layer's output (not h)
    assert np.abs(out - x["h"]).max() > 0.01


def test_items_of_one_sequence_see_each_others_new_slots():
    # two items of sequence 0 at positions 2 and 5: every K/V of the call is
    # written before any attention, so the later one reads the earlier one's
    # new slot -- the same as two calls in position order
    cfg, x = _tiny(5)
    L = x["layers"][0]
    args = (cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    h = x["h"][:2]
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    both = river.exit_layer(h, L, [2, 5], [0, 0], kc, vc, *args)
    kc2, vc2 = x["k_cache"].copy(), x["v_cache"].copy()
    first = river.exit_layer(h[:1], L, [2], [0], kc2, vc2, *args)
    second = river.exit_layer(h[1:], L, [5], [0], kc2, vc2, *args)
    np.testing.assert_allclose(both, np.concatenate([first, second]), atol=1e-13)
    np.testing.assert_allclose(kc, kc2, atol=1e-13)
    kc3, vc3 = x["k_cache"].copy(), x["v_cache"].copy()
    alone = river.exit_layer(h[1:], L, [5], [0], kc3, vc3, *args)
    assert np.abs(alone - second).max() > 1e-6   # the earlier item's slot was read


def test_own_key_score_is_rotation_free():
    # History keys 0: each earlier position scores 0. The token's own slot holds
    # RoPE(k, p) and is read by RoPE(q, p); rotations keep inner products, so its
    # score is <q, k> / sqrt(hd) from the unrotated projections, whatever p is:
    # o_h = (sum_{t<p} V[t] + e^s v) / (p + e^s). (Wd = 0: h' = h + o Wo.)
    cfg, x = _tiny(6)
    L = x["layers"][0]
    _zero(L, "d")
    j, n, hd = L["cache_layer"], len(x["h"]), cfg.head_dim
    x["k_cache"][j] = 0.0
    kc, vc = x["k_cache"].copy(), x["v_cache"].copy()
    out = river.exit_layer(x["h"], L, x["pos"], x["seq"], kc, vc, cfg.n_q_heads, cfg.n_kv_heads, hd,
                           cfg.rope_base, cfg.eps, cfg.group)
    xn = oracle.rms_norm(x["h"], L["attn_norm"], cfg.eps)
    q = (xn @ river.weight(L, "q", cfg.group)).reshape(n, cfg.n_q_heads, hd)
    k = (xn @ river.weight(L, "k", cfg.group)).reshape(n, cfg.n_kv_heads, hd)
    v = (xn @ river.weight(L, "v", cfg.group)).reshape(n, cfg.n_kv_heads, hd)
    rep = cfg.n_q_heads // cfg.n_kv_heads
    o = np.zeros((n, cfg.n_q_heads, hd))
    for i in range(n):
        p, s = x["pos"][i], x["seq"][i]
        for h in range(cfg.n_q_heads):
            g = h // rep
            e = math.exp(q[i, h] @ k[i, g] / math.sqrt(hd))
            o[i, h] = (x["v_cache"][j, s, g, :p].sum(axis=0) + e * v[i, g]) / (p + e)
    np.testing.assert_allclose(out, x["h"] + o.reshape(n, -1) @ river.weight(L, "o", cfg.group), atol=1e-11)
