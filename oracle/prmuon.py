"""fp64 restatement of one Periodic Row-wise Muon / MuonBP optimizer step.

TEST INFRASTRUCTURE ONLY (see the package docstring): plain numpy in float64,
written step by step from the method's description so that it can be checked
against the pages by eye. No blocking, fusion or reordering beyond what the
method states; numpy's matmul is the only library primitive used as a step.

Sources (cited by title and section):
  [SMDiT]   "Scaling Muon for Diffusion Transformers" -- abstract (paperdance
            card) and the PaperDaily walkthrough of the same paper, sections
            "Periodic Row-wise Muon" (Fig. 3 update rule, Fig. 4 RowNorm),
            "Distributed co-design" (Fig. 8 tall-matrix statistics) and the
            reviewer's cost note (NS5 Theta(5 r^2 c), RowNorm Theta(r c)).
  [MuonBP]  "MuonBP: Faster Muon via Block-Periodic Orthogonalization",
            abstract.

Readings taken where the pages are silent (each is also listed with its
reason in the design notes of the repository):
  * momentum is M_t = beta * M_{t-1} + G_t (no Nesterov term);
  * RowNorm normalises short-side vectors: rows when m <= n, columns when
    m > n (a square matrix counts as wide);
  * NS5 pre-normalises by the Frobenius norm plus NS_EPS, orthogonalises the
    wide orientation (tall inputs are transposed and transposed back) and uses
    X <- a X + (b A + c A A) X with A = X X^T;
  * the step size is lr on refresh / full steps and lr * gamma on RowNorm /
    block steps; decoupled weight decay multiplies W by (1 - lr * wd) with the
    base lr on every step; the shape scale defaults to sqrt(max(1, m / n));
  * MuonBP cuts each matrix into P contiguous blocks along its long side, the
    last block taking the remainder.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Sequence, Tuple

import numpy as np

# The pages never print the Newton-Schulz coefficients; this is the widely
# used quintic, taken as the library's default (a stated choice).
DEFAULT_NS_COEFFS: Tuple[float, float, float] = (3.4445, -4.7750, 2.0315)

# Added to the Frobenius norm before NS5 pre-normalisation (a stated choice;
# the pages only say the momentum is scaled before the iteration).
NS_EPS: float = 1e-7

MODE_PRMUON = 0
MODE_MUONBP = 1


def refresh_indicator(t: int, K: int) -> int:
    """rho_t of [SMDiT] section "Periodic Row-wise Muon", Fig. 3: 1 when t is a
    multiple of the period K (expensive NS5 refresh), else 0 (RowNorm step).
    MuonBP uses the same rule for its periodic full orthogonalisation
    ([MuonBP] abstract)."""
    if K < 1:
        raise ValueError("K must be >= 1")
    if t < 0:
        raise ValueError("t must be >= 0")
    return 1 if t % K == 0 else 0


def momentum_update(M_prev: np.ndarray, G: np.ndarray, beta: float) -> np.ndarray:
    """M_t = beta * M_{t-1} + G_t, in float64 ([SMDiT] abstract: the cheap
    update acts "on the current momentum"; the form itself is not printed)."""
    return beta * np.asarray(M_prev, dtype=np.float64) + np.asarray(G, dtype=np.float64)


def row_normalize(M: np.ndarray, eps: float) -> np.ndarray:
    """R_eps of [SMDiT] section "Periodic Row-wise Muon", Fig. 4: every
    short-side vector v of M is divided by max(||v||_2, eps).

    For a wide or square matrix (m <= n) the vectors are the rows, as Fig. 4
    states. For a tall matrix (m > n) they are the columns: the distributed
    section (Fig. 8) gathers per-column sums of squares nu_j for m > n, and
    both normalised maps are said to have Frobenius norm sqrt(r), r the short
    side.
    """
    M = np.asarray(M, dtype=np.float64)
    m, n = M.shape
    D = np.empty_like(M)
    if m <= n:
        for i in range(m):
            norm = math.sqrt(float(np.dot(M[i, :], M[i, :])))
            D[i, :] = M[i, :] / max(norm, eps)
    else:
        for j in range(n):
            norm = math.sqrt(float(np.dot(M[:, j], M[:, j])))
            D[:, j] = M[:, j] / max(norm, eps)
    return D


def newton_schulz(M: np.ndarray, coeffs: Sequence[float] = DEFAULT_NS_COEFFS,
                  steps: int = 5, eps_ns: float = NS_EPS) -> np.ndarray:
    """NS5 of [SMDiT] section "Periodic Row-wise Muon": approximates the polar
    factor of M by repeated matrix products and scalings, without an SVD.

    Work happens on the wide orientation (r x c, r = short side), so that the
    Gram matrix is r x r and the cost is Theta(5 r^2 c) as the reviewer's cost
    note states. Each of the `steps` iterations does
        A = X X^T,  B = b A + c A A,  X <- a X + B X.
    """
    a, b, c = (float(v) for v in coeffs)
    Y = np.asarray(M, dtype=np.float64)
    tall = Y.shape[0] > Y.shape[1]
    if tall:
        Y = Y.T
    X = Y / (np.linalg.norm(Y) + eps_ns)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tall else X


def lr_shape_scale(m: int, n: int) -> float:
    """Default per-matrix learning-rate shape scale s(m, n) = sqrt(max(1, m/n)),
    taken on the storage orientation. The pages only say the update is
    shape-scaled; this form is a stated choice, overridable per matrix."""
    return math.sqrt(max(1.0, m / n))


def apply_update(W: np.ndarray, D: np.ndarray, lr: float, wd: float,
                 eta: float, s: float) -> np.ndarray:
    """W <- W * (1 - lr * wd) - eta * s * D: decoupled weight decay (the
    walkthrough's reference [3], Loshchilov and Hutter) with the base lr,
    then the step of size eta along D."""
    W = np.asarray(W, dtype=np.float64)
    return W * (1.0 - lr * wd) - eta * s * np.asarray(D, dtype=np.float64)


def block_slices(m: int, n: int, P: int) -> List[Tuple[slice, slice]]:
    """MuonBP blocks ([MuonBP] abstract: each device orthogonalises its own
    shard): P contiguous blocks along the long side (columns when m <= n, rows
    when m > n); every block has floor(long / P) vectors except the last, which
    also takes the remainder."""
    if P < 1:
        raise ValueError("P must be >= 1")
    long_side = n if m <= n else m
    if long_side < P:
        raise ValueError("long side shorter than the number of blocks")
    base = long_side // P
    out = []
    for k in range(P):
        lo = k * base
        hi = long_side if k == P - 1 else (k + 1) * base
        if m <= n:
            out.append((slice(0, m), slice(lo, hi)))
        else:
            out.append((slice(lo, hi), slice(0, n)))
    return out


def prmuon_step(W, M_prev, G, t, K, gamma, lr, wd, beta, eps,
                coeffs=DEFAULT_NS_COEFFS, shape_scale=None):
    """One Periodic Row-wise Muon step for one matrix ([SMDiT] section
    "Periodic Row-wise Muon", Fig. 3): momentum, then NS5 on refresh steps
    (step size lr) or gamma * R_eps on the others (step size lr * gamma; gamma
    calibrates the RowNorm branch's step), then the decoupled-decay update.

    Returns (W_new, M_new, D, branch) in float64.
    """
    m, n = np.shape(M_prev)
    s = lr_shape_scale(m, n) if shape_scale is None or shape_scale <= 0 else float(shape_scale)
    M = momentum_update(M_prev, G, beta)
    rho = refresh_indicator(t, K)
    if rho:
        D = newton_schulz(M, coeffs)
        eta = lr
    else:
        D = row_normalize(M, eps)
        eta = lr * gamma
    return apply_update(W, D, lr, wd, eta, s), M, D, rho


def muonbp_step(W, M_prev, G, t, K, gamma, lr, wd, beta, eps, P,
                coeffs=DEFAULT_NS_COEFFS, shape_scale=None):
    """One MuonBP step for one matrix ([MuonBP] abstract): on full steps
    (t a multiple of K) NS5 of the whole matrix with step size lr; on the other
    steps NS5 of each of the P blocks independently, with the second step size
    lr * gamma. The shape scale is the whole matrix's.

    Returns (W_new, M_new, D, branch) in float64.
    """
    m, n = np.shape(M_prev)
    s = lr_shape_scale(m, n) if shape_scale is None or shape_scale <= 0 else float(shape_scale)
    M = momentum_update(M_prev, G, beta)
    full = refresh_indicator(t, K)
    if full:
        D = newton_schulz(M, coeffs)
        eta = lr
    else:
        D = np.empty_like(M)
        for rs, cs in block_slices(m, n, P):
            D[rs, cs] = newton_schulz(M[rs, cs], coeffs)
        eta = lr * gamma
    return apply_update(W, D, lr, wd, eta, s), M, D, full


def run_steps(Ws: Iterable[np.ndarray], Ms: Iterable[np.ndarray], grad_fn, t0: int,
              nsteps: int, K, gamma, lr, wd, beta, eps, coeffs=DEFAULT_NS_COEFFS,
              mode=MODE_PRMUON, P=8, shape_scales=None):
    """Runs `nsteps` steps t0 .. t0+nsteps-1 over a list of matrices.
    grad_fn(t, idx) returns G_t for matrix idx. Returns (Ws, Ms, branches)."""
    Ws = [np.asarray(w, dtype=np.float64).copy() for w in Ws]
    Ms = [np.asarray(mm, dtype=np.float64).copy() for mm in Ms]
    branches = []
    for t in range(t0, t0 + nsteps):
        rho = None
        for i in range(len(Ws)):
            s = None if shape_scales is None else shape_scales[i]
            G = grad_fn(t, i)
            if mode == MODE_PRMUON:
                Ws[i], Ms[i], _, rho = prmuon_step(Ws[i], Ms[i], G, t, K, gamma, lr, wd,
                                                   beta, eps, coeffs, s)
            else:
                Ws[i], Ms[i], _, rho = muonbp_step(Ws[i], Ms[i], G, t, K, gamma, lr, wd,
                                                   beta, eps, P, coeffs, s)
        branches.append(refresh_indicator(t, K) if rho is None else rho)
    return Ws, Ms, branches
