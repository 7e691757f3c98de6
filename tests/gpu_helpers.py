"""Helpers shared by the GPU parity tests: building the library, moving
tensors between the device and the fp64 oracle, error measures."""
import numpy as np
import torch

import oracle as O
from matrix_aware_optimizer_gb300 import build, synth

_built = False


def ensure_built():
    global _built
    if not _built:
        build.build_library()
        _built = True


def rel_frob(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def host64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def direction_from_update(W_prev: np.ndarray, W_new: np.ndarray, lr: float, wd: float, eta: float,
                          s: float) -> np.ndarray:
    """Solves W_new = W_prev (1 - lr wd) - eta s D for D, in fp64."""
    return (W_prev * (1.0 - lr * wd) - W_new) / (eta * s)


def make_set(shapes, grad_dtype, seed=0, device="cuda", grad_std=1e-3, param_std=0.02):
    ms = synth.MatrixSet(name="custom", shapes=tuple(shapes), grad_dtype=grad_dtype, grad_std=grad_std,
                         steps=1, seed=seed, param_std=param_std)
    return ms


def oracle_step_one(W, M, G, t, hp, mode="prmuon", P=8, s=None):
    """fp64 oracle step for one matrix from host arrays."""
    if mode == "prmuon":
        return O.prmuon_step(W, M, G, t, hp["K"], hp["gamma"], hp["lr"], hp["wd"], hp["beta"], hp["eps"],
                             shape_scale=s)
    return O.muonbp_step(W, M, G, t, hp["K"], hp["gamma"], hp["lr"], hp["wd"], hp["beta"], hp["eps"], P,
                         shape_scale=s)
