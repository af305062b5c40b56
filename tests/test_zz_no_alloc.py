"""The router gate entry point that needs no workspace, through the C ABI.

It is meant for callers that cannot allocate device memory when they call the
gate (a plugin whose host owns every device allocation, a loop where cudaMalloc
is not allowed); its scratch is an array compiled into the library. Here it
must give what the workspace entry point gives, on two calls in a row: the
second call reuses the array the first one left behind.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.parity import NEAR_BAND, SCORE_TOL
from workloads import configs, gen

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from token_early_exit_gb300 import _lib
    return _lib.load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_static_router_gate_matches_the_workspace_entry_point(lib):
    import token_early_exit_gb300 as tee
    from token_early_exit_gb300 import _lib
    cfg = configs.ROUTER_4096
    n, theta = 4096, 0.5
    w = gen.router_weights(cfg, cfg.checkpoints[1], seed=11, device=DEV)
    h = gen.router_hidden(cfg, n, cfg.checkpoints[1], seed=11, device=DEV)
    ref_score, ref_mask, ref_flag = tee.exit_gate(h, theta, w_down=w["w_down"], w_up=w["w_up"], eps=cfg.eps)
    desc = _lib.GateDesc(mode=_lib.TEE_GATE_ROUTER, rule=_lib.TEE_RULE_PER_TOKEN, dtype=_lib.TEE_BF16, d=cfg.d,
                         bottleneck=cfg.bottleneck, threshold=theta, eps=cfg.eps)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    near = (ref_score - theta).abs() <= NEAR_BAND
    for call in range(2):
        score = torch.full((n,), -1.0, device=DEV)
        mask = torch.full((n,), 7, dtype=torch.uint8, device=DEV)
        flag = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        st = lib.tee_exit_gate_router_static(ctypes.byref(desc), n, _ptr(h), h.stride(0), None, _ptr(w["w_down"]),
                                             None, _ptr(w["w_up"]), None, _ptr(score), _ptr(mask), _ptr(flag),
                                             stream)
        assert st == _lib.TEE_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert (score - ref_score).abs().max().item() <= SCORE_TOL, f"call {call}"
        assert torch.equal(mask[~near], ref_mask[~near]), f"call {call}"
        assert int(flag.item()) == int(ref_flag.item()), f"call {call}"
    # the array's sticky fault word: nothing recorded by the two clean calls
    code, detail = ctypes.c_int32(-1), ctypes.c_int32(-1)
    st = lib.tee_exit_gate_router_static_device_error(ctypes.byref(code), ctypes.byref(detail), stream)
    assert st == _lib.TEE_OK
    assert (code.value, detail.value) == (0, 0)
    assert lib.tee_exit_gate_router_static_clear_error(stream) == _lib.TEE_OK


def test_static_router_gate_rejects_sizes_beyond_its_array(lib):
    from token_early_exit_gb300 import _lib
    cfg = configs.ROUTER_4096
    desc = _lib.GateDesc(mode=_lib.TEE_GATE_ROUTER, rule=_lib.TEE_RULE_PER_TOKEN, dtype=_lib.TEE_BF16, d=cfg.d,
                         bottleneck=cfg.bottleneck, threshold=0.5, eps=cfg.eps)
    cap = lib.tee_exit_gate_router_static_max_bytes()
    n = 1 << 16   # the smallest scratch of 65,536 tokens (about 516 bytes each) is far above 4 MiB
    assert n * 512 > cap
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check answers first
    st = lib.tee_exit_gate_router_static(ctypes.byref(desc), n, fake, cfg.d, None, fake, None, fake, None, fake,
                                         fake, None, None)
    assert st == _lib.TEE_ERR_WORKSPACE
    desc.mode = _lib.TEE_GATE_COSINE
    assert lib.tee_exit_gate_router_static(ctypes.byref(desc), 8, fake, cfg.d, None, fake, None, fake, None, fake,
                                           fake, None, None) == _lib.TEE_ERR_INVALID_ARG
    assert np.isfinite(cap) and cap == 4 << 20
