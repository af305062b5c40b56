"""The C ABI library loads and exports every symbol include/tee.h declares,
and host-side argument checks answer before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from token_early_exit_gb300 import build
    build.build()
    from token_early_exit_gb300 import _lib
    return _lib.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^TEE_API\s+[\w\s\*]+?\b(tee_\w+)\s*\(", text, re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    from token_early_exit_gb300 import _lib
    names = declared_symbols()
    assert len(names) >= 16
    for name in names:
        assert hasattr(lib, name), name
    # the binding declares a signature for each of them, and for nothing else
    assert names == set(_lib.SIGNATURES)


def test_only_the_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    syms = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert syms == declared_symbols()


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.tee_version()
    assert lib.tee_status_string(0) == b"ok"
    assert lib.tee_status_string(4) == b"workspace too small"


def test_host_side_checks_need_no_gpu(lib):
    from token_early_exit_gb300 import _lib
    g = _lib.GateDesc(mode=0, rule=0, dtype=_lib.TEE_BF16, d=2048, bottleneck=0, threshold=0.97, eps=1e-5)
    assert lib.tee_exit_gate_workspace_size(ctypes.byref(g), 64) >= _lib.WS_HEADER_BYTES
    fake = ctypes.c_void_p(16)  # never dereferenced: every call below fails its checks first
    # null descriptor
    assert lib.tee_exit_gate(None, 4, fake, 2048, fake, 2048, None, None, None, None, None, fake, fake, None,
                             fake, 1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    # workspace too small
    assert lib.tee_exit_gate(ctypes.byref(g), 4, fake, 2048, fake, 2048, None, None, None, None, None, fake,
                             fake, None, fake, 8, None) == _lib.TEE_ERR_WORKSPACE
    # d not a multiple of 8
    g.d = 2047
    assert lib.tee_exit_gate(ctypes.byref(g), 4, fake, 2048, fake, 2048, None, None, None, None, None, fake,
                             fake, None, fake, 1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    # NaN threshold
    g.d, g.threshold = 2048, float("nan")
    assert lib.tee_exit_gate(ctypes.byref(g), 4, fake, 2048, fake, 2048, None, None, None, None, None, fake,
                             fake, None, fake, 1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    # misaligned row pitch (ld * 2 bytes not a multiple of 16)
    g.threshold = 0.97
    assert lib.tee_exit_gate(ctypes.byref(g), 4, fake, 2049, fake, 2048, None, None, None, None, None, fake,
                             fake, None, fake, 1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    # unsupported dtype
    g.dtype = 7
    assert lib.tee_exit_gate(ctypes.byref(g), 4, fake, 2048, fake, 2048, None, None, None, None, None, fake,
                             fake, None, fake, 1 << 20, None) == _lib.TEE_ERR_UNSUPPORTED
    # compaction: null mask / negative n / small workspace
    assert lib.tee_exit_compact(-1, fake, None, None, 0, 0, 0, fake, fake, None, None, None, 0, fake, fake,
                                1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    assert lib.tee_exit_compact(8, None, None, None, 0, 0, 0, fake, fake, None, None, None, 0, fake, fake,
                                1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    assert lib.tee_exit_compact(8, fake, None, None, 0, 0, 0, fake, fake, None, None, None, 0, fake, fake,
                                16, None) == _lib.TEE_ERR_WORKSPACE
    # scatter with d not a multiple of 8
    assert lib.tee_exit_scatter(4, fake, fake, fake, fake, 12, fake, 12, 4, 12, _lib.TEE_BF16, None, 1e-5, fake,
                                1 << 20, None) == _lib.TEE_ERR_INVALID_ARG


def test_fill_descriptor_checks(lib):
    from token_early_exit_gb300 import _lib
    D = _lib.FillDesc(d=4096, n_kv_heads=8, head_dim=128, rope_base=5e5, eps=1e-5, dtype=_lib.TEE_BF16,
                      wfmt=_lib.TEE_W_DENSE, group=64)
    assert lib.tee_kv_fill_prep_size(ctypes.byref(D), 16, 16384) > 16384 * 64 * 8
    assert lib.tee_kv_fill_workspace_size(ctypes.byref(D), 16, 14336) > 0
    D.head_dim = 7  # odd head_dim: no rotate-half pairing
    assert lib.tee_kv_fill_prep_size(ctypes.byref(D), 16, 16384) == 0
    D.head_dim, D.wfmt, D.group = 128, _lib.TEE_W_INT4, 48  # group must divide d and be a multiple of 16
    assert lib.tee_kv_fill_prep_size(ctypes.byref(D), 16, 16384) == 0
    D.group = 64
    fake = ctypes.c_void_p(16)
    layout = _lib.CacheLayout(8 * 16 * 128, 8 * 16 * 128, 16 * 128, 128, 1, 1, 8, 16)
    arr = (_lib.FillLayer * 1)()
    # workspace too small
    assert lib.tee_kv_fill(ctypes.byref(D), 1, arr, fake, 1 << 30, 4, None, fake, 4096, 4, None, None, 0, None,
                           fake, fake, ctypes.byref(layout), fake, 8, None) == _lib.TEE_ERR_WORKSPACE
    # a layer without weights
    assert lib.tee_kv_fill(ctypes.byref(D), 1, arr, fake, 1 << 30, 4, None, fake, 4096, 4, None, None, 0, None,
                           fake, fake, ctypes.byref(layout), fake, 1 << 40, None) == _lib.TEE_ERR_INVALID_ARG


def test_fused_and_ridge_entry_points_check_on_the_host(lib):
    from token_early_exit_gb300 import _lib
    fake = ctypes.c_void_p(16)  # never dereferenced: every call below fails its checks first
    # compaction + scatter: h without an output to scatter into
    assert lib.tee_exit_compact_scatter(8, fake, None, fake, 256, 256, _lib.TEE_BF16, fake, fake, None, None, None, 0,
                                        None, 0, 0, fake, fake, 1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    # gate + compaction + scatter: too small a workspace, then a misaligned output row
    g = _lib.GateDesc(mode=_lib.TEE_GATE_COSINE, rule=_lib.TEE_RULE_PER_TOKEN, dtype=_lib.TEE_BF16, d=256,
                      bottleneck=0, threshold=0.9, eps=1e-5)
    args = [ctypes.byref(g), 8, fake, 256, fake, 256, None, None, None, None, None, None, fake, fake, None, fake,
            fake, None, None, None, 0, fake, 256, 8, fake, fake]
    assert lib.tee_exit_gate_compact_scatter(*args, 8, None) == _lib.TEE_ERR_WORKSPACE
    args[22] = 257
    assert lib.tee_exit_gate_compact_scatter(*args, 1 << 20, None) == _lib.TEE_ERR_INVALID_ARG
    # ridge fit: widths off the 256-column tiles, a negative lambda, a short workspace
    assert lib.tee_ridge_fit(64, 200, 256, fake, 200, fake, 256, _lib.TEE_BF16, 0.1, fake, 256, fake, 1 << 30,
                             None) == _lib.TEE_ERR_UNSUPPORTED
    assert lib.tee_ridge_fit(64, 256, 256, fake, 256, fake, 256, _lib.TEE_BF16, -1.0, fake, 256, fake, 1 << 30,
                             None) == _lib.TEE_ERR_INVALID_ARG
    assert lib.tee_ridge_fit(64, 256, 256, fake, 256, fake, 256, _lib.TEE_BF16, 0.1, fake, 256, fake, 1024,
                             None) == _lib.TEE_ERR_WORKSPACE
    assert lib.tee_ridge_fit_workspace_size(64, 256, 256) > 256 * 256 * 4


def test_wait_timeout_check_validates_on_the_host(lib):
    from token_early_exit_gb300 import _lib
    fake = ctypes.c_void_p(16)  # never dereferenced: the calls below fail their checks first
    assert lib.tee_check_wait_timeout(None, 1000, None) == _lib.TEE_ERR_WORKSPACE
    assert lib.tee_check_wait_timeout(fake, 0, None) == _lib.TEE_ERR_INVALID_ARG
    assert lib.tee_check_wait_timeout(fake, 100001, None) == _lib.TEE_ERR_INVALID_ARG


def test_exit_river_checks_on_the_host(lib):
    from token_early_exit_gb300 import _lib
    D = _lib.RiverDesc(d=2048, n_q_heads=32, n_kv_heads=8, head_dim=64, d_ff=8192, rope_base=5e5, eps=1e-5,
                       group=64, flags=0)
    assert lib.tee_exit_river_prep_size(ctypes.byref(D), 8, 4096) > 8 * 30_000_000
    bad = _lib.RiverDesc(d=2048, n_q_heads=32, n_kv_heads=8, head_dim=96, d_ff=8192, rope_base=5e5, eps=1e-5,
                         group=64, flags=0)
    assert lib.tee_exit_river_prep_size(ctypes.byref(bad), 8, 4096) == 0   # head_dim 96 is not built
    odd = _lib.RiverDesc(d=2048, n_q_heads=30, n_kv_heads=8, head_dim=64, d_ff=8192, rope_base=5e5, eps=1e-5,
                         group=64, flags=0)
    assert lib.tee_exit_river_prep_size(ctypes.byref(odd), 8, 4096) == 0   # q heads not a multiple of kv heads
    # the attention's walk: the split walk's workspace holds the chunks' partials
    # (it grows with the cache), the pair walk's does not; other flags are refused
    by = {f: _lib.RiverDesc(d=2048, n_q_heads=32, n_kv_heads=8, head_dim=64, d_ff=8192, rope_base=5e5, eps=1e-5,
                            group=64, flags=f) for f in (_lib.TEE_RIVER_ATTN_BY_PAIR, _lib.TEE_RIVER_ATTN_BY_CHUNK, 3)}
    ws = lambda f, n, p: lib.tee_exit_river_workspace_size(ctypes.byref(by[f]), n, p)
    pair, chunk = _lib.TEE_RIVER_ATTN_BY_PAIR, _lib.TEE_RIVER_ATTN_BY_CHUNK
    assert ws(pair, 64, 4096) == ws(pair, 64, 131072) > 0
    assert ws(chunk, 64, 131072) > ws(chunk, 64, 4096) > ws(pair, 64, 4096)
    assert ws(3, 64, 4096) == 0 and lib.tee_exit_river_prep_size(ctypes.byref(by[3]), 8, 4096) == 0
    # "auto" walks pairs when n_max x n_kv_heads fills two consumer groups per SM (on any
    # part of up to 256 SMs, 64 items x 8 kv heads do; 16 items x 8 do not on one of more
    # than 64 SMs, and without a device the library assumes a full-size part)
    auto = _lib.RiverDesc(d=2048, n_q_heads=32, n_kv_heads=8, head_dim=64, d_ff=8192, rope_base=5e5, eps=1e-5,
                          group=64, flags=0)
    wa = lambda n, p: lib.tee_exit_river_workspace_size(ctypes.byref(auto), n, p)
    assert wa(128, 4096) == ws(pair, 128, 4096) and wa(128, 131072) == wa(128, 4096)
    assert wa(16, 65536) > wa(16, 4096) and wa(16, 4096) == ws(chunk, 16, 4096)
    # a cache too long for the chunk walk's merge (3 floats per query head and chunk in a
    # 32 KB buffer: 682 chunks of 256 positions at this descriptor's 4 query heads per kv
    # head) takes the pair walk even for one item
    assert wa(1, 682 * 256) == ws(chunk, 1, 682 * 256) and wa(1, 683 * 256) == ws(pair, 1, 683 * 256)
    assert wa(1, 300000) == wa(1, 600000) == ws(pair, 1, 4096)
    layout = _lib.CacheLayout(s_layer=1 << 20, s_seq=1 << 14, s_head=4096 * 64, s_pos=64, n_layers=16, n_seq=64,
                              n_heads=8, max_pos=4096)
    fake = ctypes.c_void_p(16)
    arr = (_lib.RiverLayer * 1)()
    # more than 128 items
    assert lib.tee_exit_river(ctypes.byref(D), 1, arr, fake, 1 << 30, 129, None, fake, 2048, 129, None, fake, None,
                              fake, fake, ctypes.byref(layout), fake, 2048, fake, 1 << 30, None) == \
        _lib.TEE_ERR_INVALID_ARG
    # a layer without its norm weights
    assert lib.tee_exit_river(ctypes.byref(D), 1, arr, fake, 1 << 30, 4, None, fake, 2048, 4, None, fake, None,
                              fake, fake, ctypes.byref(layout), fake, 2048, fake, 1 << 30, None) == \
        _lib.TEE_ERR_INVALID_ARG


def test_static_router_fault_query_answers_without_a_device(lib):
    # the fault word of the router gate's static array is read through the CUDA
    # runtime; with no GPU the query reports a CUDA error instead of crashing
    import torch
    from token_early_exit_gb300 import _lib
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU test reads the word")
    code, detail = ctypes.c_int32(-1), ctypes.c_int32(-1)
    assert lib.tee_exit_gate_router_static_device_error(ctypes.byref(code), ctypes.byref(detail),
                                                        None) == _lib.TEE_ERR_CUDA
    assert lib.tee_exit_gate_router_static_clear_error(None) == _lib.TEE_ERR_CUDA


def test_fill_descriptor_flags(lib):
    from token_early_exit_gb300 import _lib
    def size(flags):
        D = _lib.FillDesc(d=256, n_kv_heads=2, head_dim=64, rope_base=1e4, eps=1e-5, dtype=_lib.TEE_F32,
                          wfmt=_lib.TEE_W_DENSE, group=64, flags=flags)
        return lib.tee_kv_fill_workspace_size(ctypes.byref(D), 2, 8)
    assert size(0) > 0
    assert size(_lib.TEE_FILL_EARLY_WEIGHTS | _lib.TEE_FILL_GENERIC) == size(0)
    assert size(4) == 0   # an unknown flag is rejected


def test_decode_step_checks_on_the_host(lib):
    from token_early_exit_gb300 import _lib
    fake = ctypes.c_void_p(16)   # never dereferenced: every call below fails its checks first
    gate = _lib.GateDesc(mode=_lib.TEE_GATE_COSINE, rule=_lib.TEE_RULE_PER_TOKEN, dtype=_lib.TEE_BF16, d=2048,
                         bottleneck=0, threshold=0.97, eps=1e-5)
    fill = _lib.FillDesc(d=2048, n_kv_heads=8, head_dim=64, rope_base=5e5, eps=1e-5, dtype=_lib.TEE_BF16,
                         wfmt=_lib.TEE_W_INT4, group=64, flags=0)
    layout = _lib.CacheLayout(s_layer=1 << 20, s_seq=1 << 14, s_head=4096 * 64, s_pos=64, n_layers=16, n_seq=64,
                              n_heads=8, max_pos=4096)
    layers = (_lib.FillLayer * 1)()
    buf = _lib.StepBuffers(h_prev=16, h_cur=16, pos=16, score=16, mask=16, cont_rows=16, exit_rows=16, out=16,
                           n_out=64, counts=16, ws=16, ws_bytes=1 << 30)
    h = ctypes.c_void_p()
    # the gate's d differs from the fill's
    bad_gate = _lib.GateDesc(mode=_lib.TEE_GATE_COSINE, rule=0, dtype=_lib.TEE_BF16, d=1024, bottleneck=0,
                             threshold=0.97, eps=1e-5)
    assert lib.tee_decode_step_create(ctypes.byref(bad_gate), 64, ctypes.byref(fill), 1, layers, fake, 1 << 20, fake,
                                      fake, ctypes.byref(layout), ctypes.byref(buf), ctypes.byref(h)) == \
        _lib.TEE_ERR_INVALID_ARG
    # a workspace smaller than the calls need
    small = _lib.StepBuffers(h_prev=16, h_cur=16, pos=16, score=16, mask=16, cont_rows=16, exit_rows=16, out=16,
                             n_out=64, counts=16, ws=16, ws_bytes=256)
    assert lib.tee_decode_step_create(ctypes.byref(gate), 64, ctypes.byref(fill), 1, layers, fake, 1 << 20, fake,
                                      fake, ctypes.byref(layout), ctypes.byref(small), ctypes.byref(h)) == \
        _lib.TEE_ERR_WORKSPACE
    assert h.value is None   # set only on success
    assert lib.tee_decode_step_run_host(None, 4, fake, fake, fake, None, None, None, None, None, None) == \
        _lib.TEE_ERR_INVALID_ARG
    lib.tee_decode_step_destroy(None)
