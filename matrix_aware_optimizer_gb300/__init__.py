"""GB300-native Periodic Row-wise Muon (PR-Muon) and MuonBP optimizer step.

The compute lives in libprm.so (CUDA kernels for sm_103a behind a C ABI,
declared in include/prm.h); this package only binds it. Build the library
with `python -m matrix_aware_optimizer_gb300.build`.
"""
from . import native  # noqa: F401
from .native import PrmError, prm_branch  # noqa: F401


def __getattr__(name):
    # torch is only needed by the tensor-level API; keep `import` cheap.
    if name in ("PeriodicRowMuon", "newton_schulz", "adamw_step"):
        from . import optimizer
        return getattr(optimizer, name)
    raise AttributeError(name)
