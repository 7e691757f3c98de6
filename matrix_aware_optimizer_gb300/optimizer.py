"""torch glue over the C ABI: PyTorch supplies device memory (the tensors and
the workspace) and the stream; every arithmetic step runs in libprm."""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import native as N

_MODES = {"prmuon": N.PRM_MODE_PRMUON, "muonbp": N.PRM_MODE_MUONBP}


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class PeriodicRowMuon:
    """Periodic Row-wise Muon (and MuonBP) over a list of 2-D fp32 parameters.

    params / momenta : fp32 CUDA tensors, updated in place.
    grads            : bf16 or fp32 CUDA tensors with the same shapes (read).
    muonbp_blocks    : 0, or P > 0 to also plan MuonBP blocks.
    shape_scales     : optional per-matrix step multipliers (default
                       sqrt(max(1, rows / cols))).
    workspace_limit  : cap in bytes on the NS5 workspace: the refresh then runs
                       in sequential sub-plans that fit it. 0 (default) is the
                       library's automatic policy (whole plans up to 16 GiB,
                       4 GiB sub-plans above), -1 no cap.
    ns_form          : "auto" (default): NS5 groups wide enough to gain
                       (wide orientation r x c, c >= 1.37 r at r = 2048)
                       iterate r x r matrices in legs of at most three rounds
                       (the Gram route, ~40 % fewer flops at c = 4 r);
                       "direct": every group runs the rounds on X itself.
                       Same rounds, different rounding.
    workspace        : optional uint8 CUDA tensor to use as the scratch instead
                       of allocating one (at least workspace_bytes large).
                       Optimizers whose steps are ordered on one stream may
                       share it -- e.g. two instances over the same params and
                       momenta with two gradient buffers, alternating steps so
                       that one buffer fills while the other is consumed.
    """

    def __init__(self, params: Sequence[torch.Tensor], momenta: Sequence[torch.Tensor],
                 grads: Sequence[torch.Tensor], muonbp_blocks: int = 0,
                 shape_scales: Optional[Sequence[float]] = None, workspace_limit: int = 0,
                 workspace: Optional[torch.Tensor] = None, ns_form: str = "auto"):
        if not (len(params) == len(momenta) == len(grads)):
            raise ValueError("params, momenta and grads must have the same length")
        forms = {"auto": N.PRM_NS_FORM_AUTO, "direct": N.PRM_NS_FORM_DIRECT}
        if ns_form not in forms:
            raise ValueError(f"ns_form must be one of {sorted(forms)}")
        dev = params[0].device if params else torch.device("cuda", torch.cuda.current_device())
        if dev.type != "cuda":
            raise ValueError("tensors must live on a CUDA device")
        descs = []
        for i, (w, m, g) in enumerate(zip(params, momenta, grads)):
            if w.dim() != 2 or w.shape != m.shape or w.shape != g.shape:
                raise ValueError(f"matrix {i}: param, momentum and grad must be 2-D with one shape")
            if w.dtype != torch.float32 or m.dtype != torch.float32:
                raise ValueError(f"matrix {i}: param and momentum must be float32")
            if g.dtype not in (torch.bfloat16, torch.float32):
                raise ValueError(f"matrix {i}: grad must be bfloat16 or float32")
            for t in (w, m, g):
                if not t.is_contiguous() or t.device != dev:
                    raise ValueError(f"matrix {i}: tensors must be contiguous and on {dev}")
            d = N.prm_matrix_desc()
            d.param, d.momentum, d.grad = w.data_ptr(), m.data_ptr(), g.data_ptr()
            d.grad_dtype = N.PRM_BF16 if g.dtype == torch.bfloat16 else N.PRM_FP32
            d.rows, d.cols = w.shape
            d.shape_scale = 0.0 if shape_scales is None else float(shape_scales[i])
            descs.append(d)
        self.device = dev
        self._tensors = (list(params), list(momenta), list(grads))
        with torch.cuda.device(dev):
            self.ctx = N.prm_create(dev.index if dev.index is not None else torch.cuda.current_device())
            try:
                N.prm_set_workspace_limit(self.ctx, int(workspace_limit) if workspace_limit >= 0 else (1 << 64) - 1)
                N.prm_set_ns_form(self.ctx, forms[ns_form])
                N.prm_register_matrices(self.ctx, descs, muonbp_blocks)
                nbytes = N.prm_workspace_bytes(self.ctx)
                if workspace is None:
                    self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
                else:
                    if (workspace.dtype != torch.uint8 or workspace.device != dev or not workspace.is_contiguous()
                            or workspace.numel() < nbytes):
                        raise ValueError(f"workspace must be a contiguous uint8 tensor on {dev} "
                                         f"of at least {nbytes} bytes")
                    self.workspace = workspace
                N.prm_set_workspace(self.ctx, self.workspace.data_ptr(), self.workspace.numel())
            except Exception:
                N.prm_destroy(self.ctx)
                self.ctx = None
                raise
        self.muonbp_blocks = muonbp_blocks
        self.ns_form = ns_form

    @property
    def workspace_bytes(self) -> int:
        return self.workspace.numel()

    def step(self, t: int, K: int = 3, gamma: float = 0.15, lr: float = 0.02, wd: float = 0.01,
             beta: float = 0.95, eps: float = 1e-8, ns_coeffs=None, mode: str = "prmuon",
             stream: Optional[torch.cuda.Stream] = None) -> int:
        """Enqueues step t; returns the branch taken (1 = NS5 refresh / full)."""
        N.prm_step(self.ctx, t, K, gamma, lr, wd, beta, eps, ns_coeffs, _MODES[mode], _stream_handle(stream))
        return N.prm_branch(t, K, _MODES[mode])

    def sync_status(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        N.check(N.prm_sync_status(self.ctx, _stream_handle(stream)), "prm_sync_status", self.ctx)

    def last_direction(self, idx: int) -> torch.Tensor:
        """Direction D of the last step for matrix idx (before s * eta), as a
        CPU fp32 tensor; the momentum must still hold that step's M_t."""
        rows, cols = self._tensors[0][idx].shape
        out = torch.empty(rows, cols, dtype=torch.float32)
        N.prm_debug_last_direction(self.ctx, idx, out.data_ptr())
        return out

    def close(self) -> None:
        if getattr(self, "ctx", None) is not None:
            N.prm_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def newton_schulz(x: torch.Tensor, steps: int = 5, ns_coeffs=None,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """NS iterations of a batch of fp32 matrices [batch, m, n] (or one [m, n])
    on the tensor cores; tall matrices are orthogonalised transposed."""
    squeeze = x.dim() == 2
    xb = x.unsqueeze(0) if squeeze else x
    if xb.dtype != torch.float32 or not xb.is_cuda:
        raise ValueError("x must be a float32 CUDA tensor")
    xb = xb.contiguous()
    b, m, n = xb.shape
    out = torch.empty_like(xb)
    nbytes = N.prm_newton_schulz_workspace(b, m, n)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=xb.device)
    N.prm_newton_schulz(xb.data_ptr(), out.data_ptr(), b, m, n, ns_coeffs, steps, ws.data_ptr(), ws.numel(),
                        _stream_handle(stream))
    return out[0] if squeeze else out


def adamw_step(param: torch.Tensor, exp_avg: torch.Tensor, exp_avg_sq: torch.Tensor, grad: torch.Tensor,
               t: int, lr: float = 1e-4, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
               wd: float = 0.0, stream: Optional[torch.cuda.Stream] = None) -> None:
    """AdamW step (t >= 1) over flat fp32 CUDA tensors param / exp_avg /
    exp_avg_sq (updated in place) and a bf16 or fp32 gradient of the same
    number of elements -- the optimizer of the non-matrix parameters."""
    for x in (param, exp_avg, exp_avg_sq):
        if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
            raise ValueError("param and moments must be contiguous float32 CUDA tensors")
    if grad.dtype not in (torch.bfloat16, torch.float32) or not grad.is_contiguous():
        raise ValueError("grad must be a contiguous bfloat16 or float32 tensor")
    n = param.numel()
    if not (exp_avg.numel() == exp_avg_sq.numel() == grad.numel() == n):
        raise ValueError("all buffers must hold the same number of elements")
    N.prm_adamw_step(param.data_ptr(), exp_avg.data_ptr(), exp_avg_sq.data_ptr(), grad.data_ptr(),
                     N.PRM_BF16 if grad.dtype == torch.bfloat16 else N.PRM_FP32, n, t, lr, beta1, beta2, eps, wd,
                     _stream_handle(stream))
