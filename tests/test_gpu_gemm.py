"""Kernel-level numerics of the three tcgen05 GEMM stages of one NS5 round,
each against a plain PyTorch fp32 (CPU) computation of the same operation on
the same bf16 operands. Sizes span several tiles, partial super-blocks and a
ragged reduction tail."""
import numpy as np
import pytest
import torch

from matrix_aware_optimizer_gb300 import native as N

from .gpu_helpers import ensure_built, rel_frob

pytestmark = pytest.mark.gpu

A_C, B_C, C_C = 3.4445, -4.7750, 2.0315
SHAPES = [(3, 256, 512), (2, 384, 1000), (1, 64, 96), (2, 1024, 3072), (1, 40, 104), (4, 128, 128)]


def _pitch(x):
    return (x + 7) // 8 * 8


def _rand_bf16(batch, rows, cols, pitch, gen, scale=1.0):
    full = torch.zeros(batch, rows, pitch, dtype=torch.bfloat16)
    full[:, :, :cols] = (torch.randn(batch, rows, cols, generator=gen) * scale).to(torch.bfloat16)
    return full


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    N.load()


@pytest.mark.parametrize("batch,r,c", SHAPES)
def test_gram_matches_fp32_matmul(batch, r, c):
    gen = torch.Generator().manual_seed(r * 7 + c)
    ldc, ldr = _pitch(c), _pitch(r)
    X = _rand_bf16(batch, r, c, ldc, gen, 1.0 / np.sqrt(c))
    scale = torch.rand(batch, generator=gen) + 0.5
    Xd, sd = X.cuda(), scale.cuda()
    Ad = torch.full((batch, r, ldr), float("nan"), dtype=torch.bfloat16, device="cuda")
    N.prm_ns_gram(Xd.data_ptr(), Ad.data_ptr(), sd.data_ptr(), batch, r, c, ldc, ldr,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    A = Ad.float().cpu()[:, :, :r]
    Xf = X.float()[:, :, :c]
    ref = (scale ** 2)[:, None, None] * (Xf @ Xf.transpose(1, 2))
    for i in range(batch):
        assert torch.isfinite(A[i]).all(), "unwritten output element"
        assert rel_frob(A[i].numpy(), ref[i].numpy()) < 4e-3
    # mirrored lower triangle equals the upper one to bf16 rounding
    assert (A - A.transpose(1, 2)).abs().max().item() <= 2e-2 * A.abs().max().item()


@pytest.mark.parametrize("batch,r,c", SHAPES)
def test_poly_matches_fp32_matmul(batch, r, c):
    gen = torch.Generator().manual_seed(r * 11 + c)
    ldr = _pitch(r)
    Xs = torch.randn(batch, r, c, generator=gen) / np.sqrt(c)
    Asym = (Xs @ Xs.transpose(1, 2)).to(torch.bfloat16)
    Asym = ((Asym.float() + Asym.float().transpose(1, 2)) / 2).to(torch.bfloat16)  # exactly symmetric
    A = torch.zeros(batch, r, ldr, dtype=torch.bfloat16)
    A[:, :, :r] = Asym
    Ad = A.cuda()
    Bd = torch.full((batch, r, ldr), float("nan"), dtype=torch.bfloat16, device="cuda")
    N.prm_ns_poly(Ad.data_ptr(), Bd.data_ptr(), A_C, B_C, C_C, batch, r, ldr, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    B = Bd.float().cpu()[:, :, :r]
    Af = Asym.float()
    ref = A_C * torch.eye(r) + B_C * Af + C_C * (Af @ Af)
    for i in range(batch):
        assert torch.isfinite(B[i]).all()
        assert rel_frob(B[i].numpy(), ref[i].numpy()) < 4e-3


@pytest.mark.parametrize("batch,r,c", SHAPES)
def test_combine_matches_fp32_matmul(batch, r, c):
    gen = torch.Generator().manual_seed(r * 13 + c)
    ldc, ldr = _pitch(c), _pitch(r)
    X = _rand_bf16(batch, r, c, ldc, gen, 1.0 / np.sqrt(c))
    Braw = torch.randn(batch, r, r, generator=gen) / np.sqrt(r)
    Bsym = ((Braw + Braw.transpose(1, 2)) / 2 + A_C * torch.eye(r)).to(torch.bfloat16)
    B = torch.zeros(batch, r, ldr, dtype=torch.bfloat16)
    B[:, :, :r] = Bsym
    scale = torch.rand(batch, generator=gen) + 0.5
    Xd, Bd, sd = X.cuda(), B.cuda(), scale.cuda()
    Od = torch.full((batch, r, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    N.prm_ns_combine(Xd.data_ptr(), Bd.data_ptr(), Od.data_ptr(), sd.data_ptr(), batch, r, c, ldc, ldr,
                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    O_ = Od.float().cpu()[:, :, :c]
    Xf = X.float()[:, :, :c]
    ref = scale[:, None, None] * (Bsym.float() @ Xf)
    for i in range(batch):
        assert torch.isfinite(O_[i]).all()
        assert rel_frob(O_[i].numpy(), ref[i].numpy()) < 4e-3


def test_combine_is_not_symmetric_in_disguise():
    """A non-symmetric B would expose an operand read transposed: the kernel
    computes B X with B's rows as the A operand."""
    gen = torch.Generator().manual_seed(5)
    r, c = 256, 512
    X = _rand_bf16(1, r, c, c, gen, 0.05)
    B = torch.triu(torch.randn(1, r, r, generator=gen) * 0.05).to(torch.bfloat16)
    Xd, Bd = X.cuda(), B.cuda()
    Od = torch.empty(1, r, c, dtype=torch.bfloat16, device="cuda")
    N.prm_ns_combine(Xd.data_ptr(), Bd.data_ptr(), Od.data_ptr(), 0, 1, r, c, c, r,
                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref = B.float() @ X.float()
    assert rel_frob(Od.float().cpu().numpy(), ref.numpy()) < 4e-3
