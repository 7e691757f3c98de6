"""The allocation-free tall RowNorm step (for callers that cannot allocate
device memory while the update runs) against the regular workspace-based
path of prm_step, on two calls in a row, against the fp64 oracle, and at the
edge of its fixed scratch array. Collected last on purpose."""

import numpy as np
import pytest
import torch

import oracle as O
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


def _rel_frob_dev(a, b):
    """Relative Frobenius error in fp64, on the device (large tensors)."""
    a64, b64 = a.double(), b.double()
    return float(torch.linalg.norm(a64 - b64) / torch.linalg.norm(b64))


def _noalloc(W, M, G, shape, stream=None):
    gcode = N.PRM_BF16 if G.dtype == torch.bfloat16 else N.PRM_FP32
    N.prm_rownorm_tall_step_noalloc(W.data_ptr(), M.data_ptr(), G.data_ptr(), gcode, shape[0], shape[1],
                                    HP["gamma"], HP["lr"], HP["wd"], HP["beta"], HP["eps"], 0.0,
                                    stream if stream is not None else torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape,gdtype", [((1000, 40), torch.float32), ((4100, 132), torch.bfloat16)])
def test_noalloc_matches_oracle_twice(shape, gdtype):
    """Two allocation-free calls in a row, each checked against
    oracle.prmuon_step on the state the call started from."""
    W, M, G = _state(shape, gdtype, seed=7 + shape[1])
    for t in (1, 2):
        W0, M0, G0 = (x.double().cpu().numpy() for x in (W, M, G))
        _noalloc(W, M, G, shape)
        torch.cuda.synchronize()
        W1, M1, _, rho = O.prmuon_step(W0, M0, G0, t, **HP)
        assert rho == 0
        assert rel_frob(M.double().cpu().numpy(), M1) <= TOL_M
        assert rel_frob(W.double().cpu().numpy(), W1) <= TOL_W


def test_noalloc_at_capacity_and_just_beyond():
    """130816 x 2048 needs exactly 511 * 2048 + 2048 = 1,048,576 scratch
    floats, the whole array: accepted, and equal to prm_step within the
    tolerances on two calls in a row. One more 256-row block (131072 x 2048)
    is refused before any launch."""
    shape = (130816, 2048)
    assert (shape[0] + 255) // 256 * shape[1] + shape[1] == 1 << 20
    W, M, G = _state(shape, torch.bfloat16, seed=5)
    W2, M2 = W.clone(), M.clone()
    opt = PeriodicRowMuon([W], [M], [G])
    for t in (1, 2):
        opt.step(t, **HP)
        _noalloc(W2, M2, G, shape)
        torch.cuda.synchronize()
        assert _rel_frob_dev(M2, M) <= TOL_M
        assert _rel_frob_dev(W2, W) <= TOL_W
    opt.close()
    del W, M, G, W2, M2
    lib = N.load()
    buf = torch.zeros(64, device="cuda")
    p = buf.data_ptr()
    assert lib.prm_rownorm_tall_step_noalloc(p, p, p, N.PRM_BF16, 131072, 2048, 0.15, 0.02, 0.01, 0.95, 1e-8, 0.0,
                                             None) == N.PRM_ERR_UNSUPPORTED
