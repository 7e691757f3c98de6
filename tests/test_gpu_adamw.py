"""Parity of the fused AdamW kernel (non-matrix parameters) with the fp64
oracle, step by step from the GPU's own state. fp32 arithmetic against fp64:
relative Frobenius error <= 1e-6 on p, m and v."""
import numpy as np
import pytest
import torch

import oracle as O
from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300.optimizer import adamw_step

from .gpu_helpers import ensure_built, host64, rel_frob

pytestmark = pytest.mark.gpu
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.05)
TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def _run(n, gdtype, offset=0, steps=3, seed=0):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    # `offset` elements of slack in front: offset 1 makes every buffer 4 bytes off 16-byte alignment
    base = [torch.randn(n + offset, generator=gen, device="cuda") * 0.02 for _ in range(1)]
    p = base[0][offset:]
    m = torch.zeros(n + offset, device="cuda")[offset:]
    v = torch.zeros(n + offset, device="cuda")[offset:]
    for t in range(1, steps + 1):
        graw = torch.randn(n + offset, generator=gen, device="cuda") * 1e-3
        g = graw.to(gdtype)[offset:]
        P0, M0, V0, G0 = host64(p), host64(m), host64(v), host64(g)
        adamw_step(p, m, v, g, t, **HP)
        torch.cuda.synchronize()
        P1, M1, V1 = O.adamw_step(P0, M0, V0, G0, t, **HP)
        assert rel_frob(host64(m), M1) <= TOL
        assert rel_frob(host64(v), V1) <= TOL
        assert rel_frob(host64(p), P1) <= TOL
        # the update itself, not just the parameter, agrees closely
        assert rel_frob(host64(p) - P0 * (1 - HP["lr"] * HP["wd"]), P1 - P0 * (1 - HP["lr"] * HP["wd"])) <= 1e-4


@pytest.mark.parametrize("n", [1, 5, 4096, 1000003])
@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32])
def test_adamw_matches_oracle(n, gdtype):
    _run(n, gdtype)


def test_adamw_unaligned_buffers_take_the_scalar_path():
    _run(4099, torch.float32, offset=1)
    _run(4099, torch.bfloat16, offset=1)


def test_adamw_argument_errors():
    x = torch.zeros(8, device="cuda")
    lib = N.load()
    p = x.data_ptr()
    assert lib.prm_adamw_step(p, p, p, p, N.PRM_FP32, 8, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, None) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_adamw_step(p, p, p, p, N.PRM_FP32, 8, 1, 1e-3, 1.0, 0.999, 1e-8, 0.0, None) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_adamw_step(None, p, p, p, N.PRM_FP32, 8, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, None) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_adamw_step(None, None, None, None, N.PRM_FP32, 0, 1, 1e-3, 0.9, 0.999, 1e-8, 0.0, None) == N.PRM_OK
