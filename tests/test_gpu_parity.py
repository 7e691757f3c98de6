"""Parity of the CUDA optimizer step (through the C ABI) with the fp64 oracle
on the same seeded inputs.

Tolerances (relative Frobenius error unless stated):
  momentum M after a step                      <= 1e-6   (fp32 fma vs fp64)
  parameter W after a RowNorm step             <= 1e-5
  RowNorm direction recovered from the update  <= 1e-4   (limited by fp32 W)
  NS5 direction (bf16 operands, fp32 accum.)   <= 2e-2
  branch schedule                               exact
Checks are teacher-forced: before every step the oracle receives the GPU's
own state, so each step is judged on its own."""
import numpy as np
import pytest
import torch

import oracle as O
from matrix_aware_optimizer_gb300 import native as N
from matrix_aware_optimizer_gb300 import synth
from matrix_aware_optimizer_gb300.optimizer import PeriodicRowMuon, newton_schulz

from .gpu_helpers import direction_from_update, ensure_built, host64, make_set, rel_frob

pytestmark = pytest.mark.gpu

TOL_M = 1e-6
TOL_W_ROWNORM = 1e-5
TOL_D_ROWNORM = 1e-4
TOL_D_NS5 = 2e-2  # every shape: short sides below 64 run their rounds in fp32


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


def _hp(ms, K=None):
    return dict(K=ms.K if K is None else K, gamma=ms.gamma, lr=ms.lr, wd=ms.wd, beta=ms.beta, eps=ms.eps)


def _run_teacher_forced(ms, steps, check_idx=None, mode="prmuon", blocks=0, ns_form="auto", K=None, hp=None,
                        coeffs=None):
    shapes = ms.shapes
    Ws, Ms = synth.make_state(ms, device="cuda")
    gdt = torch.bfloat16 if ms.grad_dtype == synth.GRAD_BF16 else torch.float32
    grads = [torch.empty(s, device="cuda", dtype=gdt) for s in shapes]
    opt = PeriodicRowMuon(Ws, Ms, grads, muonbp_blocks=blocks, ns_form=ns_form)
    opt.workspace.fill_(0xFF)  # NaN bit patterns: any read of unwritten scratch shows up
    hp = _hp(ms, K) if hp is None else hp
    okw = {} if coeffs is None else {"coeffs": coeffs}
    idx = range(len(shapes)) if check_idx is None else check_idx
    report = []
    for t in steps:
        for i, g in enumerate(grads):
            synth.make_grad(shapes[i], ms.seed, t, i, ms.grad_std, ms.grad_dtype, ms.row_sigma, device="cuda", out=g)
        torch.cuda.synchronize()
        prev = {i: (host64(Ws[i]), host64(Ms[i]), host64(grads[i])) for i in idx}
        branch = opt.step(t, mode=mode, ns_coeffs=coeffs, **hp)
        opt.sync_status()
        assert branch == O.refresh_indicator(t, hp["K"])
        for i in idx:
            W0, M0, G0 = prev[i]
            m, n = shapes[i]
            s = O.lr_shape_scale(m, n)
            if mode == "prmuon":
                W1, M1, D1, rho = O.prmuon_step(W0, M0, G0, t, **hp, **okw)
            else:
                W1, M1, D1, rho = O.muonbp_step(W0, M0, G0, t, P=blocks, **hp, **okw)
            assert rho == branch
            Wg, Mg = host64(Ws[i]), host64(Ms[i])
            eta = hp["lr"] if rho else hp["lr"] * hp["gamma"]
            Dg = direction_from_update(W0, Wg, hp["lr"], hp["wd"], eta, s)
            eM, eW, eD = rel_frob(Mg, M1), rel_frob(Wg, W1), rel_frob(Dg, D1)
            report.append((t, i, rho, eM, eW, eD))
            assert eM <= TOL_M, (t, i, eM)
            if rho == 0 and mode == "prmuon":
                assert eW <= TOL_W_ROWNORM, (t, i, eW)
                assert eD <= TOL_D_ROWNORM, (t, i, eD)
            else:
                assert eD <= TOL_D_NS5, (t, i, eD)
    opt.close()
    return report


@pytest.mark.parametrize("ns_form", ["auto", "direct"])
def test_tiny_set_six_steps(ns_form):
    """4 fp32 matrices (one tall, one ragged 128x96), K=3, 6 steps: two
    refresh cycles. Two of the shapes (64 x 256, 256 x 128) are wide enough
    for the Gram route: "auto" runs their NS5 there, "direct" on X itself."""
    rep = _run_teacher_forced(synth.MATRIX_SETS["tiny"], range(6), ns_form=ns_form)
    assert [r[2] for r in rep[::4]] == [1, 0, 0, 1, 0, 0]


@pytest.mark.parametrize("ns_form", ["auto", "direct"])
def test_dit_block_d2048_full_size(ns_form):
    """The one-DiT-block set at full size (bf16 grads): a refresh step and two
    RowNorm steps on every matrix, including the tall 8192x2048 (c = 3 r and
    c = 4 r shapes take the Gram route under "auto")."""
    _run_teacher_forced(synth.MATRIX_SETS["dit_block_d2048"], range(3), ns_form=ns_form)


def test_free_running_tiny_matches_oracle():
    """Six steps without teacher forcing: the trajectories stay close (the
    bf16 NS5 error enters W through lr * D only)."""
    ms = synth.MATRIX_SETS["tiny"]
    Ws, Ms = synth.make_state(ms, device="cuda")
    W0 = [host64(w) for w in Ws]
    grads = [torch.empty(s, device="cuda") for s in ms.shapes]
    opt = PeriodicRowMuon(Ws, Ms, grads)
    host_grads = {}
    for t in range(ms.steps):
        for i, g in enumerate(grads):
            synth.make_grad(ms.shapes[i], ms.seed, t, i, ms.grad_std, ms.grad_dtype, ms.row_sigma, device="cuda", out=g)
            host_grads[(t, i)] = host64(g)
        opt.step(t, K=ms.K, gamma=ms.gamma, lr=ms.lr, wd=ms.wd, beta=ms.beta, eps=ms.eps)
    opt.sync_status()
    Wo, Mo, br = O.run_steps(W0, [np.zeros(s) for s in ms.shapes], lambda t, i: host_grads[(t, i)], 0, ms.steps,
                             ms.K, ms.gamma, ms.lr, ms.wd, ms.beta, ms.eps)
    assert br == [1, 0, 0, 1, 0, 0]
    for i in range(len(ms.shapes)):
        assert rel_frob(host64(Ms[i]), Mo[i]) <= 1e-6
        assert rel_frob(host64(Ws[i]), Wo[i]) <= 5e-3
    opt.close()


@pytest.mark.parametrize("set_name", ["tiny", "dit_block_d2048"])
def test_vanilla_muon_k1_teacher_forced(set_name):
    """K = 1 (vanilla Muon): every step is a refresh, so each step's NS5 reads
    the momentum that the previous refresh left behind. Four consecutive
    refreshes, each checked on its own against the oracle."""
    ms = synth.MATRIX_SETS[set_name]
    rep = _run_teacher_forced(ms, range(4), K=1)
    assert all(r[2] == 1 for r in rep)


def test_vanilla_muon_k1_free_running():
    """Five K = 1 steps on the tiny set without teacher forcing, against
    oracle.run_steps(..., K=1). The momentum does not depend on W, so it must
    match to fp32 rounding; W differs from the oracle's only through the NS5
    direction errors, each within TOL_D_NS5 of the oracle's direction, which
    enter W as lr * s * (error in D): the bound below adds them up over the
    steps (decayed like W)."""
    ms = synth.MATRIX_SETS["tiny"]
    steps, K = 5, 1
    Ws, Ms = synth.make_state(ms, device="cuda")
    W0 = [host64(w) for w in Ws]
    grads = [torch.empty(s, device="cuda") for s in ms.shapes]
    opt = PeriodicRowMuon(Ws, Ms, grads)
    opt.workspace.fill_(0xFF)
    host_grads = {}
    for t in range(steps):
        for i, g in enumerate(grads):
            synth.make_grad(ms.shapes[i], ms.seed, t, i, ms.grad_std, ms.grad_dtype, ms.row_sigma, device="cuda", out=g)
            host_grads[(t, i)] = host64(g)
        assert opt.step(t, K=K, gamma=ms.gamma, lr=ms.lr, wd=ms.wd, beta=ms.beta, eps=ms.eps) == 1
    opt.sync_status()
    Wo, Mo, br = O.run_steps(W0, [np.zeros(s) for s in ms.shapes], lambda t, i: host_grads[(t, i)], 0, steps,
                             K, ms.gamma, ms.lr, ms.wd, ms.beta, ms.eps)
    assert br == [1] * steps
    decay = 1.0 - ms.lr * ms.wd
    for i, (m, n) in enumerate(ms.shapes):
        # the oracle's own directions, step by step, for the error budget
        M = np.zeros((m, n))
        bound = 0.0
        for t in range(steps):
            M = O.momentum_update(M, host_grads[(t, i)], ms.beta)
            bound = bound * decay + ms.lr * O.lr_shape_scale(m, n) * TOL_D_NS5 * np.linalg.norm(O.newton_schulz(M))
        assert rel_frob(host64(Ms[i]), Mo[i]) <= TOL_M
        err = np.linalg.norm(host64(Ws[i]) - Wo[i])
        assert err <= bound, (i, err, bound)
    opt.close()


EDGE_SHAPES = [(1, 300), (300, 1), (37, 104), (100, 40), (129, 257), (257, 129), (8, 8), (64, 4100), (2, 3)]


@pytest.mark.parametrize("gdtype", [torch.float32, torch.bfloat16])
def test_edge_shapes_directions(gdtype):
    """Ragged, degenerate and odd shapes, zero vectors and vectors below eps:
    with W = 0 and wd = 0 the update is exactly -eta s D, so D is read back
    directly."""
    gen = torch.Generator().manual_seed(3)
    eps = 1e-8
    for t, K in ((1, 3), (0, 3)):
        Ws, Ms, Gs, Gh = [], [], [], []
        for (m, n) in EDGE_SHAPES:
            G = torch.randn(m, n, generator=gen)
            if m <= n and m >= 3:
                G[1] = 0.0            # a zero row
                G[2] *= 1e-11         # a row below eps
            elif m > n and n >= 3:
                G[:, 1] = 0.0
                G[:, 2] *= 1e-11
            Gd = G.to(gdtype)
            Gh.append(Gd.double().numpy())
            Gs.append(Gd.cuda())
            Ws.append(torch.zeros(m, n, device="cuda"))
            Ms.append(torch.zeros(m, n, device="cuda"))
        opt = PeriodicRowMuon(Ws, Ms, Gs)
        opt.workspace.fill_(0xFF)
        opt.step(t, K=K, gamma=0.5, lr=0.1, wd=0.0, beta=0.9, eps=eps)
        opt.sync_status()
        for i, (m, n) in enumerate(EDGE_SHAPES):
            s = O.lr_shape_scale(m, n)
            eta = 0.1 if t % K == 0 else 0.05
            Dg = -host64(Ws[i]) / (eta * s)
            if t % K == 0:
                Do = O.newton_schulz(Gh[i])
                assert rel_frob(Dg, Do) <= TOL_D_NS5, ((m, n), rel_frob(Dg, Do))
            else:
                Do = O.row_normalize(Gh[i], eps)
                assert rel_frob(Dg, Do) <= 1e-6, ((m, n), rel_frob(Dg, Do))
                assert np.all(Dg[Do == 0] == 0)
        opt.close()


@pytest.mark.parametrize("gdtype", [torch.float32, torch.bfloat16])
def test_short_side_boundary_and_long_rows(gdtype):
    """The fp32 rounds for short sides below 64 against the tensor-core
    rounds from 64 up, at the boundary (63 and 64 in both orientations), and
    on long matrices whose column tiles outnumber the 128 chunks a matrix is
    split into (40 x 300000: 4688 tiles of 64 columns, ~37 per chunk; its
    transpose; 1 x 1000000), one refresh step each against the oracle."""
    shapes = [(63, 200), (200, 63), (64, 200), (200, 64), (40, 300000), (300000, 17), (1, 1000000)]
    gen = torch.Generator().manual_seed(23)
    Gh, Ws, Ms, Gs = [], [], [], []
    for (m, n) in shapes:
        G = (torch.randn(m, n, generator=gen) * torch.exp(torch.randn(m, 1, generator=gen) * 0.5)).to(gdtype)
        Gh.append(G.double().numpy())
        Gs.append(G.cuda())
        Ws.append(torch.zeros(m, n, device="cuda"))
        Ms.append(torch.zeros(m, n, device="cuda"))
    opt = PeriodicRowMuon(Ws, Ms, Gs)
    opt.workspace.fill_(0xFF)
    assert opt.step(0, K=3, gamma=0.15, lr=0.1, wd=0.0, beta=0.9, eps=1e-8) == 1
    opt.sync_status()
    for i, (m, n) in enumerate(shapes):
        assert N.prm_ns_route(m, n) == (2 if min(m, n) < 64 else N.prm_ns_route(m, n))
        Dg = -host64(Ws[i]) / (0.1 * O.lr_shape_scale(m, n))
        e = rel_frob(Dg, O.newton_schulz(Gh[i]))
        assert e <= TOL_D_NS5, ((m, n), e)
        if min(m, n) < 64:
            assert e <= 1e-3, ((m, n), e)  # fp32 rounds: far inside the bf16 bound
    opt.close()


@pytest.mark.parametrize("gdtype", [synth.GRAD_FP32, synth.GRAD_BF16])
def test_wide_rows_past_the_256_thread_forms(gdtype):
    """Wide rows longer than the 256-thread forms hold (12288 floats) take
    the 512-thread ones: 12292 (the first width past), 13000 and 20480 (ten
    float4 per thread, partly or fully used), 24576 (fourteen), beside
    12288 (the last 256-thread width) and 13002, a width that is not a
    multiple of 4 (the scalar form), over a refresh and two RowNorm steps
    against the oracle."""
    shapes = [(24, 13000), (16, 20480), (8, 24576), (6, 12292), (5, 12288), (7, 13002)]
    ms = make_set(shapes, gdtype, seed=29)
    _run_teacher_forced(ms, steps=[0, 1, 2])


HP_CASES = [
    # K, gamma, lr, wd, beta, eps, Newton-Schulz (a, b, c), mode, blocks
    (2, 0.3, 0.05, 0.05, 0.0, 1e-8, (1.875, -0.6, -0.275), "prmuon", 0),       # no momentum history; c < 0
    (5, 0.1, 0.01, 0.0, 0.99, 1e-6, (1.5, -0.5, 0.0), "prmuon", 0),            # long period; c = 0
    (2, 1.25, 0.016, 0.02, 0.9, 1e-8, (1.875, -0.6, -0.275), "muonbp", 4),
    (4, 0.5, 0.02, 0.01, 0.5, 1e-8, (3.4445, -4.7750, 2.0315), "muonbp", 3),
]


@pytest.mark.parametrize("K,gamma,lr,wd,beta,eps,coeffs,mode,blocks", HP_CASES)
def test_step_hyperparameters_and_ns_coefficients(K, gamma, lr, wd, beta, eps, coeffs, mode, blocks):
    """prm_step with hyper-parameters other than the defaults and with
    Newton-Schulz coefficients whose c is negative or zero (the completed
    square's other sign; POLY skipped) as well as the default, teacher-forced
    against the oracle over two refreshes and the steps between, on shapes
    that take every NS5 path: a short side below 64 (fp32 rounds), the direct
    rounds (square), the Gram route (c >= 2 r; direct rounds when c = 0), a
    tall matrix and a ragged one."""
    shapes = [(40, 300), (256, 256), (128, 512), (512, 128), (96, 80)]
    ms = make_set(shapes, synth.GRAD_BF16, seed=31)
    hp = dict(K=K, gamma=gamma, lr=lr, wd=wd, beta=beta, eps=eps)
    _run_teacher_forced(ms, steps=range(K + 1), mode=mode, blocks=blocks, hp=hp, coeffs=coeffs)


@pytest.mark.parametrize("ns_form", ["auto", "direct"])
def test_more_shape_groups_than_one_launch_holds(ns_form):
    """Nine distinct shapes make nine NS5 groups (c = 2 r: all on the Gram
    route under "auto", nine r-classes under "direct"): each GEMM stage then
    runs as two launches (up to six segments each), which must give the same
    refresh as the oracle for every matrix."""
    shapes = [(32 + 16 * k, 64 + 32 * k) for k in range(9)]
    shapes[3] = (shapes[3][1], shapes[3][0])  # one tall matrix among them
    ms = make_set(shapes, synth.GRAD_BF16, seed=17)
    _run_teacher_forced(ms, steps=[0, 1], ns_form=ns_form)


def test_muonbp_block_and_full_steps():
    """MuonBP with P = 4: block steps orthogonalise each block on its own
    (wide and tall blocks, a square parent), full steps the whole matrix."""
    shapes = [(256, 1024), (1024, 256), (384, 384), (96, 640), (200, 72)]
    gen = torch.Generator().manual_seed(9)
    for t in (1, 3):
        Gh = [torch.randn(s, generator=gen) for s in shapes]
        Ws = [torch.zeros(s, device="cuda") for s in shapes]
        Ms = [torch.zeros(s, device="cuda") for s in shapes]
        Gs = [g.cuda() for g in Gh]
        opt = PeriodicRowMuon(Ws, Ms, Gs, muonbp_blocks=4)
        opt.workspace.fill_(0xFF)
        assert opt.step(t, K=3, gamma=1.25, lr=0.016, wd=0.0, beta=0.9, eps=1e-8, mode="muonbp") == (t % 3 == 0)
        opt.sync_status()
        for i, (m, n) in enumerate(shapes):
            _, _, Do, full = O.muonbp_step(np.zeros((m, n)), np.zeros((m, n)), Gh[i].double().numpy(), t, 3, 1.25,
                                           0.016, 0.0, 0.9, 1e-8, 4)
            eta = 0.016 if full else 0.016 * 1.25
            Dg = -host64(Ws[i]) / (eta * O.lr_shape_scale(m, n))
            assert rel_frob(Dg, Do) <= TOL_D_NS5, ((m, n), t, rel_frob(Dg, Do))
        opt.close()


# Long sides that the block count does not divide: the last block takes the
# remainder, so block shapes differ within one matrix and block offsets are
# not multiples of 16 bytes (300 x 1003: 125 columns = 500 bytes; 385 x 385
# with P = 3: rows of 1540 bytes). 1003 x 301 splits into wide 125 x 301
# blocks; 96 x 645 into tall 96 x 80 blocks and a 96 x 85 one; 40 x 1001 and
# 100 x 40 have blocks with short sides below 64 (the fp32 rounds).
REMAINDER_SETS = {
    8: ((300, 1003), (1003, 301), (96, 645), (40, 1001), (100, 40)),
    3: ((385, 385), (300, 1003), (1003, 301), (100, 40)),
}


@pytest.mark.parametrize("P", [8, 3])
def test_muonbp_remainder_blocks(P):
    """MuonBP with P not dividing the long side, teacher-forced against
    oracle.muonbp_step: a full step (t = 0), two block steps (t = 1, 2) and the
    next full step (t = 3)."""
    assert all(max(shp) % P != 0 for shp in REMAINDER_SETS[P])
    ms = make_set(REMAINDER_SETS[P], synth.GRAD_BF16, seed=40 + P)
    rep = _run_teacher_forced(ms, range(4), mode="muonbp", blocks=P)
    assert [r[2] for r in rep[::len(REMAINDER_SETS[P])]] == [1, 0, 0, 1]


def test_resume_is_bitwise():
    """The optimizer state is (M, t): six steps equal three steps, a fresh
    context, and three more steps, bit for bit."""
    ms = synth.MatrixSet(name="resume", shapes=((128, 384), (384, 128), (256, 256)), grad_dtype=synth.GRAD_BF16,
                         grad_std=1e-3, steps=6)

    def run(split):
        Ws, Ms = synth.make_state(ms, device="cuda")
        grads = [torch.empty(s, device="cuda", dtype=torch.bfloat16) for s in ms.shapes]
        opt = PeriodicRowMuon(Ws, Ms, grads)
        for t in range(6):
            if t == split:
                opt.close()
                opt = PeriodicRowMuon(Ws, Ms, grads)
                opt.workspace.fill_(0xFF)  # a resumed context must not depend on old scratch
            for i, g in enumerate(grads):
                synth.make_grad(ms.shapes[i], 0, t, i, 1e-3, synth.GRAD_BF16, device="cuda", out=g)
            opt.step(t)
        opt.sync_status()
        opt.close()
        return [w.cpu() for w in Ws], [m.cpu() for m in Ms]

    a, b = run(-1), run(3)
    for x, y in zip(a[0] + a[1], b[0] + b[1]):
        assert torch.equal(x, y)


def test_standalone_newton_schulz():
    gen = torch.Generator().manual_seed(21)
    for shape in [(3, 128, 512), (2, 700, 300), (1, 33, 50)]:
        X = torch.randn(*shape, generator=gen)
        D = newton_schulz(X.cuda()).cpu().double().numpy()
        for i in range(shape[0]):
            assert rel_frob(D[i], O.newton_schulz(X[i].double().numpy())) <= TOL_D_NS5


@pytest.mark.parametrize("coeffs", [
    (3.4445, -4.7750, 2.0315),   # default quintic, c > 0
    (1.5, -0.5, 0.0),            # cubic: c = 0, the polynomial stage is skipped
    (1.875, -0.6, -0.275),       # c < 0: the square enters with a minus sign
])
@pytest.mark.parametrize("shape", [(2, 320, 400), (2, 256, 600), (2, 40, 300)])
def test_newton_schulz_coefficient_signs(coeffs, shape):
    """The library forms a I + b A + c A A as a completed square whose form
    depends on the sign of c; every branch must match the plain iteration,
    on the direct route (320 x 400), on the Gram route (256 x 600, which
    falls back to the direct rounds for c = 0) and on the fp32 rounds of a
    short side below 64 (40 x 300, the plain polynomial)."""
    gen = torch.Generator().manual_seed(5)
    X = torch.randn(*shape, generator=gen)
    D = newton_schulz(X.cuda(), ns_coeffs=coeffs).cpu().double().numpy()
    for i in range(shape[0]):
        ref = O.newton_schulz(X[i].double().numpy(), coeffs=coeffs)
        assert rel_frob(D[i], ref) <= TOL_D_NS5, (coeffs, i)


def test_argument_errors_on_device():
    w = torch.zeros(64, 128, device="cuda")
    m = torch.zeros(64, 128, device="cuda")
    g = torch.zeros(64, 128, device="cuda")
    ctx = N.prm_create(0)
    try:
        d = N.prm_matrix_desc()
        d.param, d.momentum, d.grad, d.grad_dtype, d.rows, d.cols = w.data_ptr(), m.data_ptr(), g.data_ptr(), 0, 64, 128
        with pytest.raises(N.PrmError) as e:
            N.prm_step(ctx, 0, 3, 0.15, 0.02, 0.01, 0.95, 1e-8)
        assert e.value.code == N.PRM_ERR_NOT_REGISTERED
        bad = N.prm_matrix_desc()
        bad.param, bad.momentum, bad.grad, bad.rows, bad.cols = w.data_ptr() + 4, m.data_ptr(), g.data_ptr(), 64, 128
        with pytest.raises(N.PrmError) as e:
            N.prm_register_matrices(ctx, [bad])
        assert e.value.code == N.PRM_ERR_ALIGNMENT
        N.prm_register_matrices(ctx, [d])
        with pytest.raises(N.PrmError) as e:
            N.prm_step(ctx, 0, 3, 0.15, 0.02, 0.01, 0.95, 1e-8)
        assert e.value.code == N.PRM_ERR_WORKSPACE
        ws = torch.empty(N.prm_workspace_bytes(ctx) + 256, dtype=torch.uint8, device="cuda")
        with pytest.raises(N.PrmError) as e:
            N.prm_set_workspace(ctx, ws.data_ptr() + 16, N.prm_workspace_bytes(ctx))
        assert e.value.code == N.PRM_ERR_ALIGNMENT
        N.prm_set_workspace(ctx, ws.data_ptr(), ws.numel())
        with pytest.raises(N.PrmError) as e:
            N.prm_step(ctx, 1, 3, 0.15, 0.02, 0.01, 0.95, 1e-8, mode=N.PRM_MODE_MUONBP)
        assert e.value.code == N.PRM_ERR_NOT_REGISTERED
        for bad_args in ((0, 0, 0.95, 1e-8), (-1, 3, 0.95, 1e-8), (0, 3, 1.0, 1e-8), (0, 3, 0.95, 0.0)):
            t, K, beta, eps = bad_args
            with pytest.raises(N.PrmError) as e:
                N.prm_step(ctx, t, K, 0.15, 0.02, 0.01, beta, eps)
            assert e.value.code == N.PRM_ERR_INVALID_ARG
        N.prm_step(ctx, 1, 3, 0.15, 0.02, 0.01, 0.95, 1e-8)
        assert N.prm_sync_status(ctx, 0) == N.PRM_OK
    finally:
        N.prm_destroy(ctx)


@pytest.mark.parametrize("gdtype", [torch.float32, torch.bfloat16])
def test_tall_rownorm_one_launch_ragged(gdtype):
    """The one-launch tall RowNorm in both of its forms: stripes of 128
    columns with a ragged last stripe (388 = 3 x 128 + 4 and 132 = 128 + 4
    take the register form with bf16 gradients, the bulk-copy ring with fp32
    ones; 392 = 3 x 128 + 8 and 136 = 128 + 8 the ring with either), row
    tiles of 256 with ragged last tiles (1000, 4100, 130 rows), several views
    in one launch; checked against the oracle, and bit for bit against a
    second run (the column sums are reduced in a fixed order whichever tile
    finishes a stripe)."""
    shapes = [(1000, 388), (1000, 388), (4100, 132), (130, 64), (130, 64), (1000, 392), (1000, 392), (4100, 136)]
    gen = torch.Generator().manual_seed(13)
    Gh = [torch.randn(s, generator=gen).to(gdtype) for s in shapes]
    M0 = [torch.randn(s, generator=gen) * 0.5 for s in shapes]
    W0 = [torch.randn(s, generator=gen) * 0.02 for s in shapes]
    kw = dict(K=3, gamma=0.15, lr=0.02, wd=0.01, beta=0.95, eps=1e-8)

    def run():
        Ws = [w.cuda() for w in W0]
        Ms = [m.cuda() for m in M0]
        Gs = [g.cuda() for g in Gh]
        opt = PeriodicRowMuon(Ws, Ms, Gs)
        opt.workspace.fill_(0xFF)
        assert opt.step(1, **kw) == 0
        opt.sync_status()
        opt.close()
        return [w.cpu() for w in Ws], [m.cpu() for m in Ms]

    Wa, Ma = run()
    Wb, Mb = run()
    for i, (m, n) in enumerate(shapes):
        assert torch.equal(Wa[i], Wb[i]) and torch.equal(Ma[i], Mb[i])
        W1, M1, D1, rho = O.prmuon_step(W0[i].double().numpy(), M0[i].double().numpy(),
                                        Gh[i].double().numpy(), 1, **kw)
        assert rho == 0
        assert rel_frob(Ma[i].double().numpy(), M1) <= TOL_M, i
        assert rel_frob(Wa[i].double().numpy(), W1) <= TOL_W_ROWNORM, i
        Dg = direction_from_update(W0[i].double().numpy(), Wa[i].double().numpy(), kw["lr"], kw["wd"],
                                   kw["lr"] * kw["gamma"], O.lr_shape_scale(m, n))
        assert rel_frob(Dg, D1) <= TOL_D_ROWNORM, i


@pytest.mark.parametrize("steps", [1, 2, 3, 4, 6, 7])
def test_newton_schulz_round_counts(steps):
    """Other round counts than five: the Gram route splits them into legs of
    at most three (1: one direct-style round; 4: three + one; 7: three +
    three + one, the third leg back in the first X buffer); a 320 x 400
    batch member runs the direct rounds, a 33 x 50 one the fp32 rounds."""
    gen = torch.Generator().manual_seed(100 + steps)
    for shape in [(2, 192, 640), (1, 320, 400), (2, 33, 50)]:
        X = torch.randn(*shape, generator=gen)
        D = newton_schulz(X.cuda(), steps=steps).cpu().double().numpy()
        for i in range(shape[0]):
            ref = O.newton_schulz(X[i].double().numpy(), steps=steps)
            assert rel_frob(D[i], ref) <= TOL_D_NS5, (shape, steps, i, rel_frob(D[i], ref))
