"""CPU-side checks of the C ABI: the library builds and loads, exports every
entry point include/prm.h declares, and its host-only logic (argument checks,
the branch schedule) behaves as specified. No compute call is made here."""
import ctypes
import os
import re

import pytest

import oracle as O
from matrix_aware_optimizer_gb300 import build, native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return N.load()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "prm.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"PRM_API\s+[\w\s\*]+?\b(prm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for required in ("prm_create", "prm_register_matrices", "prm_workspace_bytes", "prm_set_workspace",
                     "prm_step", "prm_destroy", "prm_last_error", "prm_branch"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert names
    for name in names:
        assert hasattr(lib, name), name
        assert name in N.SIGNATURES, f"binding lacks {name}"


def test_struct_layout_matches_header():
    # 3 pointers, 2 int32, 2 int64, 2 float
    assert ctypes.sizeof(N.prm_matrix_desc) == 56
    assert N.prm_matrix_desc.rows.offset == 32


def test_branch_schedule_matches_oracle(lib):
    for mode in (N.PRM_MODE_PRMUON, N.PRM_MODE_MUONBP):
        for K in (1, 2, 3, 4, 7):
            for t in range(0, 40):
                assert N.prm_branch(t, K, mode) == O.refresh_indicator(t, K)
    assert N.prm_branch(-1, 3, 0) == -N.PRM_ERR_INVALID_ARG
    assert N.prm_branch(0, 0, 0) == -N.PRM_ERR_INVALID_ARG
    assert N.prm_branch(0, 3, 7) == -N.PRM_ERR_INVALID_ARG
    assert N.prm_branch(2 ** 40 + 3, 3, 0) == O.refresh_indicator(2 ** 40 + 3, 3)


def test_ns_route_thresholds(lib):
    """The planner's route choice. Short sides below 64 take the fp32
    CUDA-core rounds (2). Otherwise the Gram route (1) is taken when its
    executed work for five rounds is at least 10 % below the direct rounds'
    -- from c = 1.37 r at r = 2048, c = 1.9 r for r <= 256 -- never for
    square matrices, never in the direct form; the orientation does not
    matter."""
    def first_c(r):
        return next(c for c in range(r, 4 * r) if N.prm_ns_route(r, c) == 1)
    assert first_c(2048) == 2802   # 1.368 r
    assert first_c(256) == 487     # 1.902 r
    assert first_c(64) == 122
    for (m, n) in [(2048, 8192), (8192, 2048), (2048, 6144), (5120, 20480), (768, 2048), (256, 2048), (64, 300)]:
        assert N.prm_ns_route(m, n) == 1, (m, n)
        assert N.prm_ns_route(m, n, N.PRM_NS_FORM_DIRECT) == 0
    for (m, n) in [(2048, 2048), (5120, 5120), (1536, 2048), (64, 64), (320, 400)]:
        assert N.prm_ns_route(m, n) == 0, (m, n)
    # short sides below 64 take the fp32 CUDA-core rounds in both forms
    for (m, n) in [(1, 300), (300, 1), (2, 3), (8, 8), (63, 100000), (100000, 63)]:
        assert N.prm_ns_route(m, n) == 2, (m, n)
        assert N.prm_ns_route(m, n, N.PRM_NS_FORM_DIRECT) == 2, (m, n)
    assert N.prm_ns_route(0, 5) == -N.PRM_ERR_INVALID_ARG
    assert N.prm_ns_route(5, 5, 9) == -N.PRM_ERR_INVALID_ARG


def test_null_context_calls_return_status(lib):
    assert lib.prm_step(None, 0, 3, 0.15, 0.02, 0.01, 0.95, 1e-8, None, 0, None) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_register_matrices(None, None, 0, 0) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_set_workspace(None, None, 0) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_destroy(None) == N.PRM_OK
    assert lib.prm_sync_status(None, None) == N.PRM_ERR_INVALID_ARG
    n = ctypes.c_size_t(7)
    assert lib.prm_workspace_bytes(None, ctypes.byref(n)) == N.PRM_ERR_INVALID_ARG
    assert isinstance(N.last_error(None), str)


def test_standalone_argument_checks(lib):
    # rejected before any device work
    assert lib.prm_ns_gram(None, None, None, 1.0, 0.0, N.PRM_BF16, 1, 8, 8, 8, 8, None) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_ns_gram(16, 32, None, float("nan"), 0.0, N.PRM_BF16, 1, 8, 8, 8, 8, None) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_ns_gram(16, 32, None, 1.0, 0.0, N.PRM_FP32, 1, 8, 8, 8, 8, None) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_ns_combine(16, 32, 16, None, 1, 8, 8, 8, 8, None) == N.PRM_ERR_INVALID_ARG  # aliasing
    assert lib.prm_ns_poly(16, 16, 1.0, 1.0, N.PRM_FP16, 1, 8, 8, None) == N.PRM_ERR_INVALID_ARG  # aliasing
    assert lib.prm_ns_poly(16, 32, 1.0, 1.0, N.PRM_FP16, 1, 8, 12, None) == N.PRM_ERR_ALIGNMENT  # pitch % 8
    n = ctypes.c_size_t()
    assert lib.prm_newton_schulz_workspace(0, 4, 4, ctypes.byref(n)) == N.PRM_OK and n.value == 0
    assert lib.prm_newton_schulz_workspace(2, 0, 4, ctypes.byref(n)) == N.PRM_ERR_INVALID_ARG
    assert lib.prm_newton_schulz_workspace(3, 100, 40, ctypes.byref(n)) == N.PRM_OK
    # wide orientation 40 x 100: two bf16 X buffers (pitch >= 104), two 40 x 40 (pitch >= 40) ...
    assert n.value >= 3 * 40 * 104 * 2 * 2 + 3 * 40 * 40 * 2 * 2


def test_create_without_a_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = lib.prm_create(ctypes.byref(h), 0)
    assert rc in (N.PRM_ERR_CUDA, N.PRM_ERR_INVALID_ARG)
    assert not h.value
    assert N.last_error(None)
