"""prm_debug_last_direction: the direction D of the last step, read back
through the C ABI, against the fp64 oracle's direction and against the
update the step actually applied.

  D vs oracle (teacher-forced, relative Frobenius):
    RowNorm branch                   <= 1e-5  (fp32 quotient of a 1e-6 momentum)
    NS5 branch (full or per block)   <= 2e-2  (every shape)
  D vs the applied update: W_t = W_{t-1} (1 - lr wd) - eta s D within 2 ulp of
  W_t plus 8 roundings of the step term, everywhere -- the tensor-core NS5
  direction is bf16, so any other bf16 value would move W by hundreds of such
  units; the fp32 rounds of short sides below 64 are checked the same way."""
import numpy as np
import pytest
import torch

import oracle as O
from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300 import synth
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon

from .gpu_helpers import ensure_built, host64, make_set, rel_frob

pytestmark = pytest.mark.gpu

TOL_D_ROWNORM = 1e-5
TOL_D_NS5 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def _check_applied(W0, W1, D, lr, wd, eta, s):
    """W1 (fp32, from the GPU) against W0 (1 - lr wd) - eta s D in fp32 steps."""
    f = np.float32
    decay = f(1) - f(lr) * f(wd)
    step = f(eta) * f(s)
    term = (step * D.astype(np.float32)).astype(np.float64)
    pred = W0.astype(np.float64) * np.float64(decay) - term
    ulp = np.spacing(np.abs(W1).astype(np.float32)).astype(np.float64)
    # the RowNorm kernels fold s * eta / norm into one coefficient: allow a few
    # roundings of the step term on top of W's own
    bound = 2 * ulp + 8 * 2.0 ** -24 * np.abs(term) + 1e-30
    err = np.abs(W1.astype(np.float64) - pred)
    assert np.all(err <= bound), float(np.max(err / bound))


@pytest.mark.parametrize("mode,blocks,shapes,gdt", [
    ("prmuon", 0, ((64, 64), (64, 256), (256, 128), (128, 96)), synth.GRAD_FP32),
    ("prmuon", 0, ((300, 520), (520, 300), (256, 256), (40, 1000)), synth.GRAD_BF16),
    ("muonbp", 4, ((300, 520), (520, 300), (256, 256), (40, 1000)), synth.GRAD_BF16),
    # blocks with a remainder and short sides below 64 (fp32 rounds), a tall
    # matrix cut into wide blocks
    ("muonbp", 8, ((300, 1003), (1003, 301), (40, 1001), (100, 40), (8, 8)), synth.GRAD_BF16),
    ("prmuon", 0, ((1, 300), (300, 1), (8, 8), (2, 3), (37, 104), (100, 40)), synth.GRAD_FP32),
])
def test_last_direction_matches_oracle_and_update(mode, blocks, shapes, gdt):
    ms = make_set(shapes, gdt, seed=11)
    K, gamma, lr, wd, beta, eps = 3, 0.15, 0.02, 0.01, 0.95, 1e-8
    Ws, Ms = synth.make_state(ms, device="cuda")
    tdt = torch.bfloat16 if gdt == synth.GRAD_BF16 else torch.float32
    grads = [torch.empty(s, device="cuda", dtype=tdt) for s in shapes]
    opt = PeriodicRowMuon(Ws, Ms, grads, muonbp_blocks=blocks)
    for t in range(4):  # refresh, two cheap steps, refresh
        for i, g in enumerate(grads):
            synth.make_grad(shapes[i], ms.seed, t, i, ms.grad_std, gdt, ms.row_sigma, device="cuda", out=g)
        torch.cuda.synchronize()
        prev = [(host64(Ws[i]), host64(Ms[i]), host64(grads[i])) for i in range(len(shapes))]
        rho = opt.step(t, K=K, gamma=gamma, lr=lr, wd=wd, beta=beta, eps=eps, mode=mode)
        opt.sync_status()
        for i, (m, n) in enumerate(shapes):
            W0, M0, G0 = prev[i]
            W_after, M_after = Ws[i].cpu().numpy(), Ms[i].cpu().numpy()
            D = opt.last_direction(i).numpy()
            # the call reads the state, it does not write it
            assert np.array_equal(Ws[i].cpu().numpy(), W_after) and np.array_equal(Ms[i].cpu().numpy(), M_after)
            if mode == "prmuon":
                _, _, D_ref, rho_ref = O.prmuon_step(W0, M0, G0, t, K, gamma, lr, wd, beta, eps)
            else:
                _, _, D_ref, rho_ref = O.muonbp_step(W0, M0, G0, t, K, gamma, lr, wd, beta, eps, blocks)
            assert rho_ref == rho
            ns5 = rho == 1 or mode == "muonbp"
            tol = TOL_D_NS5 if ns5 else TOL_D_ROWNORM
            e = rel_frob(D, D_ref)
            assert e <= tol, (mode, t, i, e)
            eta = np.float32(lr) if rho == 1 else np.float32(lr) * np.float32(gamma)
            _check_applied(prev[i][0].astype(np.float32), W_after, D, lr, wd, eta, O.lr_shape_scale(m, n))
    opt.close()


def test_last_direction_errors():
    shapes = ((64, 128),)
    ms = make_set(shapes, synth.GRAD_FP32, seed=3)
    Ws, Ms = synth.make_state(ms, device="cuda")
    grads = [torch.zeros(s, device="cuda") for s in shapes]
    opt = PeriodicRowMuon(Ws, Ms, grads)
    with pytest.raises(N.PrmError):
        opt.last_direction(0)  # no step yet
    opt.step(0)
    opt.sync_status()
    out = torch.empty(64, 128)
    with pytest.raises(N.PrmError):
        N.prm_debug_last_direction(opt.ctx, 1, out.data_ptr())
    with pytest.raises(N.PrmError):
        N.prm_debug_last_direction(opt.ctx, -1, out.data_ptr())
    with pytest.raises(N.PrmError):
        N.prm_debug_last_direction(opt.ctx, 0, 0)
    # zero momentum: NS5 of 0 is 0
    assert torch.count_nonzero(opt.last_direction(0)) == 0
    opt.close()
