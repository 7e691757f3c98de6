"""Parity at the benchmark's full sizes, in the benchmark's launch
configuration (every matrix of the set registered in one context), on
sampled outputs the fp64 oracle can compute one by one:
  * RowNorm steps: sampled short-side vectors of every shape (a row of a wide
    matrix, a column of a tall one, depends only on itself);
  * refresh / MuonBP steps: whole sampled matrices, one per shape.
Tolerances are those of the parity tests."""
import numpy as np
import pytest
import torch

import oracle as O
from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300 import synth
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon

from .gpu_helpers import direction_from_update, ensure_built, host64, rel_frob

pytestmark = pytest.mark.gpu

TOL_M = 1e-6
TOL_W_ROWNORM = 1e-5
TOL_D_ROWNORM = 1e-4
TOL_D_NS5 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def _first_of_each_shape(shapes):
    seen, idx = set(), []
    for i, s in enumerate(shapes):
        if s not in seen:
            seen.add(s)
            idx.append(i)
    return idx


def _setup(ms):
    dev = torch.device("cuda")
    Ws, Ms = synth.make_state(ms, device=dev)
    gdt = torch.bfloat16 if ms.grad_dtype == synth.GRAD_BF16 else torch.float32
    grads = [torch.empty(s, device=dev, dtype=gdt) for s in ms.shapes]
    opt = PeriodicRowMuon(Ws, Ms, grads, muonbp_blocks=ms.blocks)
    return Ws, Ms, grads, opt


def _fill_grads(ms, grads, t):
    for i, g in enumerate(grads):
        synth.make_grad(ms.shapes[i], ms.seed, t, i, ms.grad_std, ms.grad_dtype, ms.row_sigma, device="cuda", out=g)


def _sample_vectors(shape, k, rng):
    m, n = shape
    return np.sort(rng.choice(m if m <= n else n, size=min(k, min(m, n)), replace=False))


def _check_rownorm_sampled(ms, Ws, Ms, grads, opt, t, rng, k=8):
    hp = dict(K=ms.K, gamma=ms.gamma, lr=ms.lr, wd=ms.wd, beta=ms.beta, eps=ms.eps)
    samples = {}
    for i, s in enumerate(ms.shapes):
        if i % 7 and i != len(ms.shapes) - 1:
            continue  # a spread of matrices, always including the last
        sel = _sample_vectors(s, k, rng)
        ti = torch.as_tensor(sel, device="cuda")
        wide = s[0] <= s[1]
        take = (lambda x: x.index_select(0, ti)) if wide else (lambda x: x.index_select(1, ti))
        samples[i] = (sel, wide, host64(take(Ws[i])), host64(take(Ms[i])), host64(take(grads[i])))
    assert opt.step(t, **hp) == 0
    opt.sync_status()
    for i, (sel, wide, W0, M0, G0) in samples.items():
        ti = torch.as_tensor(sel, device="cuda")
        take = (lambda x: x.index_select(0, ti)) if wide else (lambda x: x.index_select(1, ti))
        m, n = ms.shapes[i]
        s = O.lr_shape_scale(m, n)
        # one row (column) at a time: R_eps is local to a short-side vector
        for j in range(len(sel)):
            sl = (slice(j, j + 1), slice(None)) if wide else (slice(None), slice(j, j + 1))
            W1, M1, D1, rho = O.prmuon_step(W0[sl], M0[sl], G0[sl], t, shape_scale=s, **hp)
            assert rho == 0
            Wg, Mg = host64(take(Ws[i]))[sl], host64(take(Ms[i]))[sl]
            assert rel_frob(Mg, M1) <= TOL_M
            assert rel_frob(Wg, W1) <= TOL_W_ROWNORM
            Dg = direction_from_update(W0[sl], Wg, ms.lr, ms.wd, ms.lr * ms.gamma, s)
            assert rel_frob(Dg, D1) <= TOL_D_ROWNORM


def _check_ns_sampled(ms, Ws, Ms, grads, opt, t, idx, mode="prmuon"):
    hp = dict(K=ms.K, gamma=ms.gamma, lr=ms.lr, wd=ms.wd, beta=ms.beta, eps=ms.eps)
    prev = {i: (host64(Ws[i]), host64(Ms[i]), host64(grads[i])) for i in idx}
    branch = opt.step(t, mode=mode, **hp)
    opt.sync_status()
    for i in idx:
        W0, M0, G0 = prev[i]
        if mode == "prmuon":
            W1, M1, D1, rho = O.prmuon_step(W0, M0, G0, t, **hp)
        else:
            W1, M1, D1, rho = O.muonbp_step(W0, M0, G0, t, P=ms.blocks, **hp)
        assert rho == branch
        m, n = ms.shapes[i]
        eta = ms.lr if rho else ms.lr * ms.gamma
        Dg = direction_from_update(W0, host64(Ws[i]), ms.lr, ms.wd, eta, O.lr_shape_scale(m, n))
        assert rel_frob(host64(Ms[i]), M1) <= TOL_M
        assert rel_frob(Dg, D1) <= TOL_D_NS5, (i, (m, n), rel_frob(Dg, D1))


def test_dit_1p3b_sampled():
    """1.3B-shaped set (97 matrices, 1.23 G parameters): a refresh step with
    NS5 checked on one matrix of every shape, then two RowNorm steps checked on
    sampled rows / columns across the set."""
    ms = synth.MATRIX_SETS["dit_1p3b"]
    Ws, Ms, grads, opt = _setup(ms)
    rng = np.random.default_rng(0)
    _fill_grads(ms, grads, 0)
    _check_ns_sampled(ms, Ws, Ms, grads, opt, 0, _first_of_each_shape(ms.shapes))
    for t in (1, 2):
        _fill_grads(ms, grads, t)
        _check_rownorm_sampled(ms, Ws, Ms, grads, opt, t, rng)
    opt.close()
    del Ws, Ms, grads, opt
    torch.cuda.empty_cache()


def test_dit_1p3b_muonbp_sampled():
    """MuonBP on the 1.3B set (8 blocks per matrix, 776 blocks): a full step
    and a block step, checked on one matrix of every shape."""
    ms = synth.MATRIX_SETS["dit_1p3b_muonbp"]
    Ws, Ms, grads, opt = _setup(ms)
    idx = _first_of_each_shape(ms.shapes)
    for t in (0, 1):
        _fill_grads(ms, grads, t)
        _check_ns_sampled(ms, Ws, Ms, grads, opt, t, idx, mode="muonbp")
    opt.close()
    del Ws, Ms, grads, opt
    torch.cuda.empty_cache()


def test_dit_15b_sampled():
    """15B-shaped set (192 matrices, 15.1 G parameters, ~151 GB of state plus
    the NS5 workspace): RowNorm steps on sampled vectors of every shape, and
    the NS5 refresh checked on the square 5120 x 5120 matrix and on a tall
    20480 x 5120 one (orthogonalised transposed; ~1.2e13 fp64 FLOPs in the
    oracle)."""
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < 215e9:
        pytest.skip("needs ~215 GB of free device memory")
    ms = synth.MATRIX_SETS["dit_15b"]
    Ws, Ms, grads, opt = _setup(ms)
    rng = np.random.default_rng(1)
    _fill_grads(ms, grads, 0)
    _check_ns_sampled(ms, Ws, Ms, grads, opt, 0, [1, 3])
    _fill_grads(ms, grads, 1)
    _check_rownorm_sampled(ms, Ws, Ms, grads, opt, 1, rng, k=4)
    opt.close()
    del Ws, Ms, grads, opt
    torch.cuda.empty_cache()
