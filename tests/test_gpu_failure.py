"""Failure detection on the GPU without a fault: a bounded device-side wait
is made to run out on a flag that nothing sets, and the error reaches the
host while the context stays usable.

The one-launch tall RowNorm kernel's update tiles wait for their column
stripe's inverse norms (a flag the stripe's last momentum tile publishes).
prm_debug_withhold_tall_norms keeps one stripe's flag unpublished for one
step: its update tiles give up after the given limit and leave that stripe
of W unchanged; the other stripe is updated as the oracle says, the
momentum everywhere; prm_sync_status reports PRM_ERR_TIMEOUT once, and the
next step runs clean."""
import numpy as np
import pytest
import torch

import oracle as O
from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon

from .gpu_helpers import ensure_built, host64, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def test_withheld_stripe_times_out_and_context_recovers():
    m, n = 1024, 256  # tall: two stripes of 128 columns
    gen = torch.Generator().manual_seed(4)
    W0 = torch.randn(m, n, generator=gen) * 0.02
    M0 = torch.randn(m, n, generator=gen) * 1e-3
    G = torch.randn(m, n, generator=gen) * 1e-3
    W, M, Gd = W0.cuda(), M0.cuda(), G.cuda()
    opt = PeriodicRowMuon([W], [M], [Gd])
    kw = dict(K=3, gamma=0.15, lr=0.02, wd=0.01, beta=0.95, eps=1e-8)
    N.prm_debug_withhold_tall_norms(opt.ctx, 1, 0.05)
    assert opt.step(1, **kw) == 0
    with pytest.raises(N.PrmError) as e:
        opt.sync_status()
    assert e.value.code == N.PRM_ERR_TIMEOUT
    W1, M1 = host64(W), host64(M)
    Wr, Mr, _, _ = O.prmuon_step(W0.double().numpy(), M0.double().numpy(), G.double().numpy(), 1, **kw)
    assert rel_frob(M1, Mr) <= 1e-6                       # the momentum pass completed
    assert np.array_equal(W1[:, 128:], W0.double().numpy()[:, 128:])  # the withheld stripe: untouched
    assert rel_frob(W1[:, :128], Wr[:, :128]) <= 1e-5     # the other stripe: updated
    # one report only, and the context keeps working
    opt.sync_status()
    opt.step(2, **kw)
    opt.sync_status()
    W2, M2 = host64(W), host64(M)
    Wr2, Mr2, _, _ = O.prmuon_step(W1, M1, G.double().numpy(), 2, **kw)
    assert rel_frob(M2, Mr2) <= 1e-6 and rel_frob(W2, Wr2) <= 1e-5
    opt.close()


def test_withhold_arguments():
    W = torch.zeros(256, 128, device="cuda")
    opt = PeriodicRowMuon([W], [torch.zeros_like(W)], [torch.zeros_like(W)])
    for stripe, limit in ((-1, 0.1), (0, 0.0), (0, 2.5)):
        with pytest.raises(N.PrmError) as e:
            N.prm_debug_withhold_tall_norms(opt.ctx, stripe, limit)
        assert e.value.code == N.PRM_ERR_INVALID_ARG
    # armed, then a refresh step: no effect there, it waits for the next RowNorm step
    N.prm_debug_withhold_tall_norms(opt.ctx, 0, 0.05)
    opt.step(0)
    opt.sync_status()
    opt.step(1)
    with pytest.raises(N.PrmError):
        opt.sync_status()
    opt.close()
