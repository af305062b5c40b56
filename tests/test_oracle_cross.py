"""The C++ oracle against the independent numpy restatement of the same
definitions (``oracle.numpy_ref``), function by function, on random inputs.

Both compute in float64; the C++ sums run in index order with plain loops,
numpy's through BLAS in its own order, so floating-point results agree to a
few ulps of the values' scale and integer results exactly. Neither side is
the pin of the other (those are the closed forms, invariants and worked
examples of tests/test_oracle_*.py); this checks that no entry point of the
C++ library drifts from its definition in a way only some inputs reveal."""
import subprocess

import numpy as np
import pytest

import oracle
from oracle import numpy_ref as ref
from oracle import river
from oracle.numpy_ref import river as ref_river
from tests.parity import host
from workloads import configs, gen

RNG = np.random.default_rng(7)
TOL = dict(rtol=1e-11, atol=1e-12)


def _same(a, b):
    for x, y in zip(a if isinstance(a, tuple) else (a,), b if isinstance(b, tuple) else (b,)):
        if isinstance(x, (int, np.integer)) or np.asarray(x).dtype.kind in "iub":
            assert np.array_equal(np.asarray(x), np.asarray(y))
        else:
            np.testing.assert_allclose(x, y, **TOL)


@pytest.mark.parametrize("rule", ["per_token", "batch_all"])
def test_cosine_gate(rule):
    a = RNG.standard_normal((37, 96))
    b = 0.9 * a + 0.3 * RNG.standard_normal((37, 96))
    b[5] = 0.0   # a zero row
    _same(oracle.cosine_gate(a, b, 0.93, rule), ref.cosine_gate(a, b, 0.93, rule))
    _same(oracle.cosine_gate(a, a, 0.5, rule), ref.cosine_gate(a, a, 0.5, rule))


@pytest.mark.parametrize("extras", [False, True])
def test_router_gate(extras):
    n, d, b = 29, 64, 16
    h = RNG.standard_normal((n, d))
    wd, wu = 0.2 * RNG.standard_normal((b, d)), 0.5 * RNG.standard_normal(b)
    kw = dict(gamma=1 + 0.1 * RNG.standard_normal(d), b_down=RNG.standard_normal(b), b_up=0.3) if extras else {}
    for rule in ("per_token", "batch_all"):
        _same(oracle.router_gate(h, wd, wu, 0.5, rule, eps=1e-5, **kw),
              ref.router_gate(h, wd, wu, 0.5, rule, eps=1e-5, **kw))


def test_earliest_exit_and_layer_ops():
    probs = {k: RNG.uniform(0, 1, 50) for k in (3, 7, 11, 15)}
    for k_min in (0, 8):
        d1 = oracle.earliest_exit(probs, 0.7, 16, k_min)
        assert np.array_equal(d1, ref.earliest_exit(probs, 0.7, 16, k_min))
        assert oracle.layer_ops(d1) == ref.layer_ops(d1)


def test_compaction_and_scatter():
    n, d = 45, 24
    mask = (RNG.uniform(size=n) < 0.4).astype(np.uint8)
    pos_in = RNG.permutation(100)[:n]
    p1, p2 = oracle.stable_partition(mask, pos_in), ref.stable_partition(mask, pos_in)
    for k in p2:
        assert np.array_equal(p1[k], p2[k]), k
    h = RNG.standard_normal((n, d))
    _same(oracle.gather_rows(h, p1["cont_rows"]), ref.gather_rows(h, p2["cont_rows"]))
    out = RNG.standard_normal((100, d))
    g = 1 + 0.1 * RNG.standard_normal(d)
    _same(oracle.exit_scatter(out, h, p1["exit_rows"], p1["exit_pos"]),
          ref.exit_scatter(out, h, p2["exit_rows"], p2["exit_pos"]))
    _same(oracle.exit_scatter(out, h, p1["exit_rows"], p1["exit_pos"], gamma=g, eps=1e-5),
          ref.exit_scatter(out, h, p2["exit_rows"], p2["exit_pos"], gamma=g, eps=1e-5))


def test_dequant_norm_rope():
    packed = RNG.integers(0, 256, (64, 24), dtype=np.uint8)
    s, z = RNG.uniform(0.01, 0.1, (2, 24)), RNG.uniform(4, 11, (2, 24))
    _same(oracle.dequant_int4(packed, s, z, 64), ref.dequant_int4(packed, s, z, 64))
    x = RNG.standard_normal((3, 5, 32))
    g = RNG.standard_normal(32)
    _same(oracle.rms_norm(x, g, 1e-5), ref.rms_norm(x, g, 1e-5))
    pos = RNG.integers(0, 120000, (3, 1))
    _same(oracle.rope_rotate_half(x, pos, 5e5), ref.rope_rotate_half(x, pos, 5e5))


@pytest.mark.parametrize("variant", ["dense_map", "identity_int4", "bias_norm"])
def test_fill(variant):
    t, d, nkv, hd = 9, 128, 2, 32
    kvw = nkv * hd
    L = {"gamma": 1 + 0.1 * RNG.standard_normal(d), "cache_layer": 1, "w_map": None}
    if variant == "identity_int4":
        for c in "kv":
            L[f"w{c}"] = RNG.integers(0, 256, (d // 2, kvw), dtype=np.uint8)
            L[f"{c}_scale"] = RNG.uniform(0.01, 0.05, (d // 64, kvw))
            L[f"{c}_zero"] = RNG.uniform(6, 9, (d // 64, kvw))
    else:
        L["wk"], L["wv"] = RNG.standard_normal((d, kvw)) / 20, RNG.standard_normal((d, kvw)) / 20
    if variant == "dense_map":
        L["w_map"] = RNG.standard_normal((d, d)) / 11 + 0.5 * np.eye(d)
    if variant == "bias_norm":
        L["k_bias"], L["v_bias"], L["k_norm"] = RNG.standard_normal(kvw), RNG.standard_normal(kvw), \
            1 + 0.2 * RNG.standard_normal(hd)
    h = RNG.standard_normal((t, d))
    pos = RNG.integers(0, 4096, t)
    _same(oracle.fill_rows(h, L, pos, nkv, hd, 1e4, 1e-5), ref.fill_rows(h, L, pos, nkv, hd, 1e4, 1e-5))
    kc = RNG.standard_normal((2, 3, nkv, 4096, hd))
    rows, seq = np.array([4, 0, 7]), RNG.integers(0, 3, t)
    _same(oracle.kv_fill(h, [L], kc, kc, nkv, hd, 1e4, 1e-5, rows=rows, pos=pos, seq=seq),
          ref.kv_fill(h, [L], kc, kc, nkv, hd, 1e4, 1e-5, rows=rows, pos=pos, seq=seq))


def test_ridge():
    X, Y = RNG.standard_normal((80, 24)), RNG.standard_normal((80, 10))
    np.testing.assert_allclose(oracle.ridge_fit(X, Y, 0.3), ref.ridge_fit(X, Y, 0.3), rtol=1e-9, atol=1e-12)


def test_exit_river():
    cfg = configs.TINY_RIVER
    x = host(gen.river_inputs(cfg, 3))
    a = RNG.standard_normal(40) * 4
    _same(river.silu(a), ref_river.silu(a))
    q = RNG.standard_normal((4, cfg.n_q_heads, cfg.head_dim))
    kl, vl = x["k_cache"][0], x["v_cache"][0]
    pos, seq = x["pos"][:4], x["seq"][:4]
    _same(river.attention(q, kl, vl, pos, seq, cfg.n_kv_heads), ref_river.attention(q, kl, vl, pos, seq,
                                                                                    cfg.n_kv_heads))
    args = (cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps, cfg.group)
    kc1, vc1 = x["k_cache"].copy(), x["v_cache"].copy()
    kc2, vc2 = x["k_cache"].copy(), x["v_cache"].copy()
    o1 = river.exit_river(x["h"], x["layers"], x["pos"], x["seq"], kc1, vc1, *args)
    o2 = ref_river.exit_river(x["h"], x["layers"], x["pos"], x["seq"], kc2, vc2, *args)
    np.testing.assert_allclose(o1, o2, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(kc1, kc2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(vc1, vc2, rtol=1e-10, atol=1e-12)


def test_oracle_library_is_plain_single_threaded_code():
    # it links nothing but the C/C++ runtime (no BLAS, no OpenMP) and starts no thread
    from oracle import _native
    _native.lib()
    libs = subprocess.run(["ldd", _native.LIB], capture_output=True, text=True).stdout.lower()
    assert not any(w in libs for w in ("blas", "lapack", "gomp", "omp", "tbb", "mkl")), libs
    und = subprocess.run(["nm", "-D", "--undefined-only", _native.LIB], capture_output=True, text=True).stdout
    assert "pthread_create" not in und and "dgemm" not in und
