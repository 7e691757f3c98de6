"""fp64 restatement of one AdamW step, for the non-matrix parameters.

TEST INFRASTRUCTURE ONLY (see the package docstring). "Scaling Muon for
Diffusion Transformers" (PaperDaily walkthrough, section on the scaling study)
keeps biases, normalisation parameters and other non-matrix parameters on
AdamW; its reference [3] (Loshchilov and Hutter, decoupled weight decay) is
the method. The pages print no formula, so the plain reading of that
reference is taken: Adam's bias-corrected first and second moments, and a
weight decay applied to the parameter directly (not through the gradient):

  m <- b1 m + (1 - b1) g            v <- b2 v + (1 - b2) g^2
  m_hat = m / (1 - b1^t)            v_hat = v / (1 - b2^t)
  p <- p (1 - lr wd) - lr m_hat / (sqrt(v_hat) + eps)

with t = 1 on the first step.
"""
from __future__ import annotations

import numpy as np


def adamw_step(p, m, v, g, t, lr, beta1, beta2, eps, wd):
    """One AdamW step at 1-based step count t. Returns (p, m, v) in float64."""
    if t < 1:
        raise ValueError("t counts steps from 1")
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v
