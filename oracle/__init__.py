"""Plain fp64 CPU oracle for the Periodic Row-wise Muon (PR-Muon) and MuonBP
optimizer step.

This package is TEST INFRASTRUCTURE. It is the yardstick the CUDA library is
checked against, never a part of it: only the test suite, the package smoke
check and the benchmark's CPU-baseline leg may import it. It shares no code
with the GPU path (no kernels, helpers, tables or constants); the two meet only
through the seeded input generators, which hold none of the method's
arithmetic.
"""
from .prmuon import (  # noqa: F401
    DEFAULT_NS_COEFFS,
    NS_EPS,
    refresh_indicator,
    momentum_update,
    row_normalize,
    newton_schulz,
    lr_shape_scale,
    apply_update,
    block_slices,
    prmuon_step,
    muonbp_step,
    run_steps,
)
from .adamw import adamw_step  # noqa: F401,E402
