"""The allocation-free tall RowNorm step (for callers that cannot allocate
device memory while the update runs) against the regular workspace-based
path of prm_step, on two calls in a row. Collected last on purpose."""

import pytest
import torch

from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon

from .gpu_helpers import ensure_built, rel_frob

pytestmark = pytest.mark.gpu

TOL_M = 1e-6   # the momentum tolerance of the parity tests
TOL_W = 1e-5   # the RowNorm-step parameter tolerance of the parity tests
HP = dict(K=3, gamma=0.15, lr=0.02, wd=0.01, beta=0.95, eps=1e-8)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def _state(shape, gdtype, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    W = torch.randn(shape, generator=gen, device="cuda") * 0.02
    M = torch.randn(shape, generator=gen, device="cuda") * 1e-3
    rows = torch.exp(torch.randn((shape[0], 1), generator=gen, device="cuda") * 0.5)
    G = (torch.randn(shape, generator=gen, device="cuda") * rows * 1e-3).to(gdtype)
    return W, M, G


@pytest.mark.parametrize("shape,gdtype", [((8192, 2048), torch.bfloat16), ((1000, 40), torch.float32),
                                          ((300, 1), torch.bfloat16)])
def test_noalloc_matches_workspace_path_twice(shape, gdtype):
    W, M, G = _state(shape, gdtype, seed=shape[0] + shape[1])
    W2, M2 = W.clone(), M.clone()
    opt = PeriodicRowMuon([W], [M], [G])
    stream = torch.cuda.current_stream().cuda_stream
    gcode = N.PRM_BF16 if gdtype == torch.bfloat16 else N.PRM_FP32
    for t in (1, 2):  # two RowNorm steps in a row (t % K != 0)
        opt.step(t, **HP)
        N.prm_rownorm_tall_step_noalloc(W2.data_ptr(), M2.data_ptr(), G.data_ptr(), gcode, shape[0], shape[1],
                                        HP["gamma"], HP["lr"], HP["wd"], HP["beta"], HP["eps"], 0.0, stream)
        torch.cuda.synchronize()
        assert rel_frob(M2.double().cpu().numpy(), M.double().cpu().numpy()) <= TOL_M
        assert rel_frob(W2.double().cpu().numpy(), W.double().cpu().numpy()) <= TOL_W
    opt.close()


def test_noalloc_rejects_what_it_cannot_hold():
    lib = N.load()
    buf = torch.zeros(64, device="cuda")
    p = buf.data_ptr()
    # 200000 x 2048 would need 782 * 2048 + 2048 scratch floats (> 1 Mi): refused before any launch
    assert lib.prm_rownorm_tall_step_noalloc(p, p, p, N.PRM_FP32, 200000, 2048, 0.15, 0.02, 0.01, 0.95, 1e-8, 0.0,
                                             None) == N.PRM_ERR_UNSUPPORTED
    assert lib.prm_rownorm_tall_step_noalloc(p, p, p, N.PRM_FP32, 64, 64, 0.15, 0.02, 0.01, 0.95, 1e-8, 0.0,
                                             None) == N.PRM_ERR_SHAPE
    assert lib.prm_rownorm_tall_step_noalloc(None, p, p, N.PRM_FP32, 64, 8, 0.15, 0.02, 0.01, 0.95, 1e-8, 0.0,
                                             None) == N.PRM_ERR_INVALID_ARG
