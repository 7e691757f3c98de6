"""Seeded synthetic inputs for the optimizer step: parameters, zero momentum and
per-step gradients with the shapes of the DiT matrix sets.

This module only draws random numbers; it holds none of the optimizer's
arithmetic, so the CUDA library and its fp64 CPU checker can both be fed from
it. Values are drawn with torch's generator on the requested device (CUDA
generation is what makes the multi-GB sets cheap to build); the CPU checker
receives copies of the very same tensors.

Workload recipe (shapes from the DiT matrix sets of "Scaling Muon for
Diffusion Transformers", 1.3B and 15B scales):
  * parameters W ~ N(0, 0.02^2), fp32;
  * momentum starts at zero, fp32;
  * gradients G = N(0, sigma^2) * exp(N(0, 0.5^2)) with one log-normal scale per
    storage row (sigma = 1 for the tiny fp32 set, 1e-3 in bf16 for the DiT
    sets); a fresh gradient per (step, matrix).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import torch

GRAD_FP32 = "fp32"
GRAD_BF16 = "bf16"


@dataclass(frozen=True)
class MatrixSet:
    """A named workload: matrix shapes plus the step's hyper-parameters."""
    name: str
    shapes: Tuple[Tuple[int, int], ...]
    grad_dtype: str
    grad_std: float
    steps: int
    K: int = 3
    gamma: float = 0.15
    lr: float = 0.02
    wd: float = 0.01
    beta: float = 0.95
    eps: float = 1e-8
    mode: str = "prmuon"
    blocks: int = 0
    row_sigma: float = 0.5
    param_std: float = 0.02
    seed: int = 0
    description: str = field(default="", compare=False)

    @property
    def params(self) -> int:
        return sum(m * n for m, n in self.shapes)


def _dit_block(d: int, up: int, adaln: Optional[int]):
    blk = [(d, 3 * d), (d, d), (d, up), (up, d)]
    return blk, ([(d, adaln)] if adaln else [])


def _dit_set(d: int, nblocks: int, adaln: Optional[int]):
    blk, extra = _dit_block(d, 4 * d, adaln)
    return tuple(blk * nblocks + extra)


MATRIX_SETS: Dict[str, MatrixSet] = {
    "tiny": MatrixSet(
        name="tiny",
        shapes=((64, 64), (64, 256), (256, 128), (128, 96)),
        grad_dtype=GRAD_FP32, grad_std=1.0, steps=6,
        description="4 fp32 matrices 64x64, 64x256, 256x128 (tall), 128x96; 6 steps"),
    "dit_block_d2048": MatrixSet(
        name="dit_block_d2048",
        shapes=((2048, 6144), (2048, 2048), (2048, 8192), (8192, 2048), (2048, 12288)),
        grad_dtype=GRAD_BF16, grad_std=1e-3, steps=12,
        description="one DiT block at d=2048: qkv, attn-out, mlp-up, mlp-down (tall), adaLN"),
    "dit_1p3b": MatrixSet(
        name="dit_1p3b",
        shapes=_dit_set(2048, 24, 12288),
        grad_dtype=GRAD_BF16, grad_std=1e-3, steps=30,
        description="1.3B-shaped DiT matrix set: 24 blocks at d=2048 + shared adaLN 2048x12288"),
    "dit_1p3b_4blk": MatrixSet(
        name="dit_1p3b_4blk",
        shapes=_dit_set(2048, 4, None),
        grad_dtype=GRAD_BF16, grad_std=1e-3, steps=30,
        description="4 blocks of the 1.3B-shaped set (16 matrices, 2.4 GB of state): a profiling case "
                    "whose launches have the full set's per-group shape but a few GB on the device"),
    "dit_1p3b_muonbp": MatrixSet(
        name="dit_1p3b_muonbp",
        shapes=_dit_set(2048, 24, 12288),
        grad_dtype=GRAD_BF16, grad_std=1e-3, steps=30,
        mode="muonbp", blocks=8, lr=0.02 * 0.8, gamma=1.25,
        description="MuonBP on the 1.3B set: 8 blocks per matrix along the long side; "
                    "lr_block=0.02 (block steps), lr_full=0.016 (every 3rd step)"),
    "dit_1p3b_4blk_muonbp": MatrixSet(
        name="dit_1p3b_4blk_muonbp",
        shapes=_dit_set(2048, 4, None),
        grad_dtype=GRAD_BF16, grad_std=1e-3, steps=30,
        mode="muonbp", blocks=8, lr=0.02 * 0.8, gamma=1.25,
        description="MuonBP on 4 blocks of the 1.3B-shaped set: a profiling case with the full "
                    "set's block shapes (768, 256 and 1024 x 2048 NS5 groups) on a few GB"),
    "dit_1p3b_mlp_up": MatrixSet(
        name="dit_1p3b_mlp_up",
        shapes=((8192, 2048),) * 24,
        grad_dtype=GRAD_BF16, grad_std=1e-3, steps=30,
        description="the 24 tall mlp-up matrices of the 1.3B-shaped set (402.7 M params): a profiling "
                    "case for the tall RowNorm kernel"),
    "dit_15b": MatrixSet(
        name="dit_15b",
        shapes=_dit_set(5120, 48, None),
        grad_dtype=GRAD_BF16, grad_std=1e-3, steps=9,
        description="15B-shaped DiT matrix set: 48 blocks at d=5120"),
}

def dit_vector_params(d: int, nblocks: int, adaln: Optional[int]) -> int:
    """Number of non-matrix parameters of the DiT sets (left to AdamW): per
    block the biases of qkv (3d), attention out (d), mlp up (4d) and down
    (d) plus two normalisation layers' scale and shift (4d); the shared
    adaLN modulation's bias when there is one."""
    return nblocks * 13 * d + (adaln or 0)


_KIND = {"param": 1, "grad": 2, "rowscale": 3}


def stream_seed(base: int, kind: str, t: int, idx: int) -> int:
    """Deterministic 63-bit seed for one (kind, step, matrix) draw."""
    x = (base * 0x9E3779B97F4A7C15 + _KIND[kind] * 0xBF58476D1CE4E5B9
         + (t + 1) * 0x94D049BB133111EB + (idx + 1) * 0x2545F4914F6CDD1D)
    return x & 0x7FFFFFFFFFFFFFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_param(shape, seed: int, idx: int, std: float = 0.02, device="cpu") -> torch.Tensor:
    """W ~ N(0, std^2), fp32."""
    g = _gen(device, stream_seed(seed, "param", 0, idx))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def make_grad(shape, seed: int, t: int, idx: int, std: float, dtype: str,
              row_sigma: float = 0.5, device="cpu", out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """G = N(0, std^2) * exp(N(0, row_sigma^2)) per storage row; fp32 or bf16."""
    m, n = shape
    g = _gen(device, stream_seed(seed, "grad", t, idx))
    base = torch.randn((m, n), generator=g, device=device, dtype=torch.float32)
    gs = _gen(device, stream_seed(seed, "rowscale", t, idx))
    rows = torch.exp(torch.randn((m, 1), generator=gs, device=device, dtype=torch.float32) * row_sigma)
    base.mul_(rows).mul_(std)
    tdt = torch.bfloat16 if dtype == GRAD_BF16 else torch.float32
    if out is not None:
        out.copy_(base)
        return out
    return base.to(tdt)


def make_state(ms: MatrixSet, device="cpu", shapes=None):
    """(params, momenta) lists for a matrix set: W ~ N(0, 0.02^2), M = 0."""
    shapes = ms.shapes if shapes is None else shapes
    Ws = [make_param(s, ms.seed, i, ms.param_std, device) for i, s in enumerate(shapes)]
    Ms = [torch.zeros(s, device=device, dtype=torch.float32) for s in shapes]
    return Ws, Ms


def make_grads(ms: MatrixSet, t: int, device="cpu", shapes=None) -> List[torch.Tensor]:
    shapes = ms.shapes if shapes is None else shapes
    return [make_grad(s, ms.seed, t, i, ms.grad_std, ms.grad_dtype, ms.row_sigma, device)
            for i, s in enumerate(shapes)]
