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
# the completed-square stage constants of the default quintic
GRAM_GAIN = np.sqrt(C_C)
GRAM_DIAG = B_C / (2 * np.sqrt(C_C))
POLY_GAIN = 1.0
POLY_DIAG = A_C - B_C ** 2 / (4 * C_C)
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


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("batch,r,c", SHAPES)
def test_gram_matches_fp32_matmul(batch, r, c, out_dtype):
    gen = torch.Generator().manual_seed(r * 7 + c)
    ldc, ldr = _pitch(c), _pitch(r)
    X = _rand_bf16(batch, r, c, ldc, gen, 1.0 / np.sqrt(c))
    scale = torch.rand(batch, generator=gen) + 0.5
    Xd, sd = X.cuda(), scale.cuda()
    Ad = torch.full((batch, r, ldr), float("nan"), dtype=out_dtype, device="cuda")
    N.prm_ns_gram(Xd.data_ptr(), Ad.data_ptr(), sd.data_ptr(), GRAM_GAIN, GRAM_DIAG,
                  N.PRM_FP16 if out_dtype == torch.float16 else N.PRM_BF16, batch, r, c, ldc, ldr,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    A = Ad.float().cpu()[:, :, :r]
    Xf = X.float()[:, :, :c]
    ref = GRAM_GAIN * (scale ** 2)[:, None, None] * (Xf @ Xf.transpose(1, 2)) + GRAM_DIAG * torch.eye(r)
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
    # C = sqrt(c) A + b / (2 sqrt(c)) I, stored in fp16 as the Gram stage writes it
    C = GRAM_GAIN * (Xs @ Xs.transpose(1, 2)) + GRAM_DIAG * torch.eye(r)
    Asym = ((C + C.transpose(1, 2)) / 2).to(torch.float16)  # exactly symmetric
    A = torch.zeros(batch, r, ldr, dtype=torch.float16)
    A[:, :, :r] = Asym
    Ad = A.cuda()
    Bd = torch.full((batch, r, ldr), float("nan"), dtype=torch.bfloat16, device="cuda")
    N.prm_ns_poly(Ad.data_ptr(), Bd.data_ptr(), POLY_GAIN, POLY_DIAG, N.PRM_FP16, batch, r, ldr,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    B = Bd.float().cpu()[:, :, :r]
    Af = Asym.float()
    ref = POLY_GAIN * (Af @ Af) + POLY_DIAG * torch.eye(r)
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


@pytest.mark.parametrize("gain", [1.0, -1.0])
def test_poly_negative_gain(gain):
    """sgn(c) = -1 (a quintic with c < 0) flips the square's sign."""
    gen = torch.Generator().manual_seed(9)
    r = 384
    Xs = torch.randn(1, r, 512, generator=gen) / np.sqrt(512)
    Csym = (Xs @ Xs.transpose(1, 2) - 0.5 * torch.eye(r)).to(torch.bfloat16)
    Csym = ((Csym.float() + Csym.float().transpose(1, 2)) / 2).to(torch.bfloat16)
    Cd = Csym.cuda()
    Pd = torch.empty_like(Cd)
    N.prm_ns_poly(Cd.data_ptr(), Pd.data_ptr(), gain, 0.25, N.PRM_BF16, 1, r, r,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    Cf = Csym.float()
    ref = gain * (Cf @ Cf) + 0.25 * torch.eye(r)
    assert rel_frob(Pd.float().cpu().numpy(), ref.numpy()) < 4e-3
