"""A capped workspace splits the refresh into sequential sub-plans; the
result must not change (bit for bit: each matrix's kernels see the same
data whatever batch it shares), in PR-Muon and MuonBP mode. Optimizers
whose steps share a stream may also share one workspace."""
import pytest
import torch

from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300 import synth
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon

from .gpu_helpers import ensure_built, make_set

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


SHARE_A = ((256, 768), (768, 256), (40, 300), (4096, 128))
SHARE_B = ((512, 512), (8192, 256), (300, 40), (128, 1536))


def _run_pair(shared):
    sets = [make_set(SHARE_A, synth.GRAD_BF16, seed=41), make_set(SHARE_B, synth.GRAD_BF16, seed=42)]
    state = [synth.make_state(ms, device="cuda") for ms in sets]
    grads = [[torch.empty(s, device="cuda", dtype=torch.bfloat16) for s in ms.shapes] for ms in sets]
    ws = None
    if shared:
        need = []
        for (Ws, Ms), g in zip(state, grads):
            probe = PeriodicRowMuon(Ws, Ms, g)
            need.append(probe.workspace_bytes)
            probe.close()
        ws = torch.empty(max(need), dtype=torch.uint8, device="cuda")
        with pytest.raises(ValueError):
            PeriodicRowMuon(state[0][0], state[0][1], grads[0], workspace=ws[:min(need) // 2])
    opts = [PeriodicRowMuon(Ws, Ms, g, workspace=ws) for (Ws, Ms), g in zip(state, grads)]
    for t in range(4):
        for k, ms in enumerate(sets):
            for i, g in enumerate(grads[k]):
                synth.make_grad(ms.shapes[i], ms.seed, t, i, 1e-3, synth.GRAD_BF16, device="cuda", out=g)
            opts[k].step(t, K=3, gamma=0.15)  # the two optimizers' steps alternate on one stream
    out = []
    for opt, (Ws, Ms) in zip(opts, state):
        opt.sync_status()
        opt.close()
        out += [w.cpu() for w in Ws] + [m.cpu() for m in Ms]
    return out


def test_optimizers_sharing_one_workspace():
    """Optimizers whose steps run on one stream may share one scratch buffer
    (`workspace=`, at least each one's workspace_bytes): alternating
    refreshes and RowNorm steps (tall ones included) give bit for bit the
    W and M of the same optimizers with buffers of their own, and a buffer
    smaller than needed is refused."""
    own = _run_pair(shared=False)
    shared = _run_pair(shared=True)
    for x, y in zip(own, shared):
        assert torch.equal(x, y)
