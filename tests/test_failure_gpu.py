"""Failure detection on the GPU without a fault: the bounded wait that every
pipeline of the library uses gives up on a barrier that nothing completes,
records a time-out in the workspace header and returns, and the context stays
usable for the next call."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def test_bounded_wait_records_a_timeout_and_returns(tee):
    ws = tee.Workspace(DEV)
    t0 = time.perf_counter()
    ws.check_wait_timeout(2000)   # 2 ms
    code, detail = ws.device_error()   # synchronises
    assert time.perf_counter() - t0 < 5.0
    assert (code, detail) == (6, 99)   # TEE_DEVERR_TIMEOUT, where = the check's wait
    ws.clear_error()
    assert ws.device_error() == (0, 0)
    # the context is usable: an exit gate afterwards gives its exact answer
    h = torch.randn(64, 256, device=DEV)
    score, mask, flag = tee.exit_gate(h, 0.5, h_prev=h, ws=ws)
    torch.cuda.synchronize()
    assert torch.allclose(score, torch.ones_like(score), atol=1e-5)
    assert bool((mask == 1).all()) and int(flag.item()) == 1
    assert ws.device_error() == (0, 0)


def test_the_first_fault_is_kept(tee):
    ws = tee.Workspace(DEV)
    ws.check_wait_timeout(500)
    ws.check_wait_timeout(500)
    assert ws.device_error() == (6, 99)
