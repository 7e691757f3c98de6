"""A whole K=3 PR-Muon (or MuonBP) cycle captured into a CUDA graph and
replayed gives bit-for-bit the same state as running the steps directly:
prm_step only enqueues kernels and asynchronous memsets on the caller's
stream, and the branch of each position in the cycle is fixed by t mod K."""
import pytest
import torch

from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300 import synth
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon

from .gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def _setup():
    ms = synth.MatrixSet(name="graph", shapes=((256, 768), (768, 256), (512, 512), (100, 40)),
                         grad_dtype=synth.GRAD_BF16, grad_std=1e-3, steps=9)
    Ws, Ms = synth.make_state(ms, device="cuda")
    grads = [synth.make_grad(s, 0, 0, i, 1e-3, synth.GRAD_BF16, device="cuda") for i, s in enumerate(ms.shapes)]
    return ms, Ws, Ms, grads


@pytest.mark.parametrize("mode,blocks", [("prmuon", 0), ("muonbp", 4)])
def test_graph_replay_matches_direct_steps(mode, blocks):
    ms, Wa, Ma, ga = _setup()
    opt_a = PeriodicRowMuon(Wa, Ma, ga, muonbp_blocks=blocks)
    for t in range(9):
        opt_a.step(t, mode=mode)
    opt_a.sync_status()

    ms, Wb, Mb, gb = _setup()
    opt_b = PeriodicRowMuon(Wb, Mb, gb, muonbp_blocks=blocks)
    # first cycle directly (also warms up per-device set-up), then capture one cycle
    for t in range(3):
        opt_b.step(t, mode=mode)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side):
        for t in range(3, 6):
            opt_b.step(t, mode=mode)
    # capture records without executing: two replays run cycles 2 and 3
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    opt_b.sync_status()
    for x, y in zip(Wa + Ma, Wb + Mb):
        assert torch.equal(x, y)
    opt_a.close()
    opt_b.close()
