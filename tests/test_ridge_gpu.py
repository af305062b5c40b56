"""RidgeFill's closed-form map fitted on the GPU (tee_ridge_fit) against the
oracle's float64 Cholesky solve on the same bf16 calibration rows."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def tee():
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as t
    return t


def _rows(n, d, d_out, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    x = torch.randn(n, d, device=DEV, generator=g)
    a = torch.randn(d, d_out, device=DEV, generator=g) / d ** 0.5 + 0.5 * torch.eye(d, d_out, device=DEV)
    y = x @ a + 0.1 * torch.randn(n, d_out, device=DEV, generator=g)
    return x.to(torch.bfloat16), y.to(torch.bfloat16)


@pytest.mark.parametrize("n,d,d_out,lam", [(1024, 256, 256, 0.1), (3000, 512, 256, 1.0), (700, 256, 512, 5.0),
                                           (4096, 1024, 1024, 0.5)])
def test_ridge_fit_matches_the_oracle(tee, n, d, d_out, lam):
    x, y = _rows(n, d, d_out, seed=n + d)
    ws = tee.Workspace(DEV)
    w = tee.ridge_fit(x, y, lam, ws=ws)
    torch.cuda.synchronize()
    assert ws.device_error() == (0, 0)
    ref = oracle.ridge_fit(f64(x), f64(y), lam)
    got = w.double().cpu().numpy()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-3, rel
    assert np.abs(got - ref).max() <= 1e-3 * np.abs(ref).max() + 1e-4


def test_ridge_fit_recovers_the_map_as_lambda_vanishes(tee):
    # Y = X A exactly (X and A in {-1, 0, 1}: every entry of Y an integer of at most
    # 256 in magnitude, exact in bf16): the fit returns A up to the fp32 solve and
    # the O(lambda) bias
    n, d = 2048, 256
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    x = torch.randint(-1, 2, (n, d), device=DEV, generator=g).float()
    a = torch.randint(-1, 2, (d, d), device=DEV, generator=g).float()
    y = x @ a
    assert torch.equal(y.to(torch.bfloat16).float(), y)
    w = tee.ridge_fit(x.to(torch.bfloat16), y.to(torch.bfloat16), 1e-4)
    torch.cuda.synchronize()
    assert float((w - a).abs().max()) <= 2e-3


def test_ridge_fit_records_a_non_positive_pivot(tee):
    n, d = 256, 256
    x = torch.zeros(n, d, device=DEV, dtype=torch.bfloat16)   # X^T X = 0 and lambda = 0
    y = torch.ones(n, d, device=DEV, dtype=torch.bfloat16)
    ws = tee.Workspace(DEV)
    w = tee.ridge_fit(x, y, 0.0, ws=ws)
    torch.cuda.synchronize()
    code, detail = ws.device_error()
    assert code == 7 and detail == 0
    assert bool(torch.isnan(w).any())
