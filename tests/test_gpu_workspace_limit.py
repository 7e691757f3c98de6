"""A capped workspace splits the refresh into sequential sub-plans; the
result must not change (bit for bit: each matrix's kernels see the same
data whatever batch it shares), in PR-Muon and MuonBP mode."""
import pytest
import torch

from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300 import synth
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon

from .gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu

# the last two shapes have short sides below 64 (fp32 rounds), in whole
# matrices and, with P = 4, in their MuonBP blocks
SHAPES = ((256, 768),) * 5 + ((768, 256),) * 5 + ((512, 512),) * 4 + ((384, 1024),) * 2 + ((40, 700),) * 3 + \
    ((900, 24),) * 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def _run(limit, mode, blocks):
    ms = synth.MatrixSet(name="cap", shapes=SHAPES, grad_dtype=synth.GRAD_BF16, grad_std=1e-3, steps=4)
    Ws, Ms = synth.make_state(ms, device="cuda")
    grads = [torch.empty(s, device="cuda", dtype=torch.bfloat16) for s in SHAPES]
    opt = PeriodicRowMuon(Ws, Ms, grads, muonbp_blocks=blocks, workspace_limit=limit)
    nbytes = opt.workspace_bytes
    for t in range(4):
        for i, g in enumerate(grads):
            synth.make_grad(SHAPES[i], 0, t, i, 1e-3, synth.GRAD_BF16, device="cuda", out=g)
        opt.step(t, mode=mode, K=3, gamma=1.25 if mode == "muonbp" else 0.15)
    opt.sync_status()
    opt.close()
    return [w.cpu() for w in Ws] + [m.cpu() for m in Ms], nbytes


@pytest.mark.parametrize("mode,blocks", [("prmuon", 0), ("muonbp", 4)])
def test_capped_workspace_gives_identical_results(mode, blocks):
    full, full_bytes = _run(-1, mode, blocks)  # no cap: one plan
    auto, auto_bytes = _run(0, mode, blocks)   # automatic: a set this small stays whole
    assert auto_bytes == full_bytes
    for x, y in zip(full, auto):
        assert torch.equal(x, y)
    cap = full_bytes // 5
    capped, capped_bytes = _run(cap, mode, blocks)
    assert capped_bytes < full_bytes
    assert capped_bytes <= max(cap, 256)
    for x, y in zip(full, capped):
        assert torch.equal(x, y)
