"""ctypes binding of libprm (include/prm.h): the same entry points under the
same names, argument marshalling only. Every step of the optimizer runs in the
library's CUDA kernels; there is no Python or CPU fallback, and loading fails
loudly when the shared library has not been built."""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_uint16, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libprm.so")

PRM_OK = 0
PRM_ERR_INVALID_ARG = 1
PRM_ERR_SHAPE = 2
PRM_ERR_ALIGNMENT = 3
PRM_ERR_NOT_REGISTERED = 4
PRM_ERR_CUDA = 5
PRM_ERR_TIMEOUT = 6
PRM_ERR_OOM = 7
PRM_ERR_WORKSPACE = 8
PRM_ERR_UNSUPPORTED = 9

PRM_FAMILY_ROWNORM_WIDE = 0
PRM_FAMILY_ROWNORM_TALL = 1
PRM_FAMILY_NS_PREP = 2
PRM_FAMILY_NS_GRAM = 3
PRM_FAMILY_NS_POLY = 4
PRM_FAMILY_NS_COMBINE = 5
FAMILY_NAMES = ["rownorm_wide", "rownorm_tall", "ns_prep", "ns_gram", "ns_poly", "ns_combine", "ns_sym",
                "ns_small"]

PRM_FP32 = 0
PRM_BF16 = 1
PRM_FP16 = 2
PRM_MODE_PRMUON = 0
PRM_MODE_MUONBP = 1
PRM_NS_FORM_AUTO = 0
PRM_NS_FORM_DIRECT = 1

ERROR_NAMES = {
    PRM_OK: "OK", PRM_ERR_INVALID_ARG: "INVALID_ARG", PRM_ERR_SHAPE: "SHAPE",
    PRM_ERR_ALIGNMENT: "ALIGNMENT", PRM_ERR_NOT_REGISTERED: "NOT_REGISTERED", PRM_ERR_CUDA: "CUDA",
    PRM_ERR_TIMEOUT: "TIMEOUT", PRM_ERR_OOM: "OOM", PRM_ERR_WORKSPACE: "WORKSPACE",
    PRM_ERR_UNSUPPORTED: "UNSUPPORTED",
}


class prm_matrix_desc(ctypes.Structure):
    _fields_ = [
        ("param", c_void_p),
        ("momentum", c_void_p),
        ("grad", c_void_p),
        ("grad_dtype", c_int32),
        ("reserved", c_int32),
        ("rows", c_int64),
        ("cols", c_int64),
        ("shape_scale", c_float),
        ("reserved2", c_float),
    ]


# name -> (restype, argtypes), mirroring include/prm.h
SIGNATURES = {
    "prm_create": (c_int, [POINTER(c_void_p), c_int]),
    "prm_destroy": (c_int, [c_void_p]),
    "prm_register_matrices": (c_int, [c_void_p, POINTER(prm_matrix_desc), c_int, c_int]),
    "prm_workspace_bytes": (c_int, [c_void_p, POINTER(c_size_t)]),
    "prm_set_workspace_limit": (c_int, [c_void_p, c_size_t]),
    "prm_set_ns_form": (c_int, [c_void_p, c_int]),
    "prm_ns_route": (c_int, [c_int64, c_int64, c_int]),
    "prm_debug_withhold_tall_norms": (c_int, [c_void_p, c_int, ctypes.c_double]),
    "prm_set_workspace": (c_int, [c_void_p, c_void_p, c_size_t]),
    "prm_step": (c_int, [c_void_p, c_int64, c_int, c_float, c_float, c_float, c_float, c_float,
                         POINTER(c_float), c_int, c_void_p]),
    "prm_branch": (c_int, [c_int64, c_int, c_int]),
    "prm_sync_status": (c_int, [c_void_p, c_void_p]),
    "prm_debug_last_direction": (c_int, [c_void_p, c_int, c_void_p]),
    "prm_last_error": (c_char_p, [c_void_p]),
    "prm_profile": (c_int, [c_void_p, c_int]),
    "prm_profile_read": (c_int, [c_void_p, c_int, POINTER(ctypes.c_double), POINTER(c_int64), POINTER(c_int64),
                                 POINTER(ctypes.c_double)]),
    "prm_ns_gram": (c_int, [c_void_p, c_void_p, c_void_p, c_float, c_float, c_int, c_int, c_int64, c_int64,
                            c_int64, c_int64, c_void_p]),
    "prm_ns_poly": (c_int, [c_void_p, c_void_p, c_float, c_float, c_int, c_int, c_int64, c_int64, c_void_p]),
    "prm_ns_combine": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int64, c_int64, c_int64,
                               c_int64, c_void_p]),
    "prm_rownorm_tall_step_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int64, c_int64, c_float,
                                              c_float, c_float, c_float, c_float, c_float, c_void_p]),
    "prm_adamw_step": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int64, c_int64, ctypes.c_double,
                               ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double, c_void_p]),
    "prm_newton_schulz_workspace": (c_int, [c_int, c_int64, c_int64, POINTER(c_size_t)]),
    "prm_newton_schulz": (c_int, [c_void_p, c_void_p, c_int, c_int64, c_int64, POINTER(c_float), c_int,
                                  c_void_p, c_size_t, c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libprm.so (once) and declares every entry point's signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libprm.so not found at {path}: build it first "
            "(python -m matrix_aware_optimizer_gb300.build, or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class PrmError(RuntimeError):
    def __init__(self, code: int, where: str, message: str = ""):
        self.code = code
        super().__init__(f"{where} failed with PRM_ERR_{ERROR_NAMES.get(code, code)}"
                         + (f": {message}" if message else ""))


def last_error(ctx) -> str:
    msg = load().prm_last_error(ctx)
    return msg.decode() if msg else ""


def check(code: int, where: str, ctx=None) -> None:
    if code != PRM_OK:
        raise PrmError(code, where, last_error(ctx))


# thin same-name wrappers ------------------------------------------------------
def prm_create(device: int = 0):
    h = c_void_p()
    check(load().prm_create(ctypes.byref(h), device), "prm_create", None)
    return h


def prm_destroy(ctx) -> None:
    check(load().prm_destroy(ctx), "prm_destroy")


def prm_register_matrices(ctx, descs, muonbp_blocks: int = 0) -> None:
    arr = (prm_matrix_desc * max(1, len(descs)))(*descs)
    check(load().prm_register_matrices(ctx, arr, len(descs), muonbp_blocks), "prm_register_matrices", ctx)


def prm_set_workspace_limit(ctx, max_bytes: int) -> None:
    check(load().prm_set_workspace_limit(ctx, max_bytes), "prm_set_workspace_limit", ctx)


def prm_set_ns_form(ctx, form: int) -> None:
    check(load().prm_set_ns_form(ctx, form), "prm_set_ns_form", ctx)


def prm_ns_route(m: int, n: int, form: int = PRM_NS_FORM_AUTO) -> int:
    return load().prm_ns_route(m, n, form)


def prm_workspace_bytes(ctx) -> int:
    n = c_size_t()
    check(load().prm_workspace_bytes(ctx, ctypes.byref(n)), "prm_workspace_bytes", ctx)
    return n.value


def prm_set_workspace(ctx, ptr: int, nbytes: int) -> None:
    check(load().prm_set_workspace(ctx, c_void_p(ptr), nbytes), "prm_set_workspace", ctx)


def _coeff_ptr(coeffs):
    if coeffs is None:
        return None
    return (c_float * 3)(*[float(c) for c in coeffs])


def prm_step(ctx, t: int, K: int, gamma: float, lr: float, wd: float, beta: float, eps: float,
             ns_coeffs=None, mode: int = PRM_MODE_PRMUON, stream: int = 0) -> None:
    check(load().prm_step(ctx, t, K, gamma, lr, wd, beta, eps, _coeff_ptr(ns_coeffs), mode,
                          c_void_p(stream)), "prm_step", ctx)


def prm_branch(t: int, K: int, mode: int = PRM_MODE_PRMUON) -> int:
    return load().prm_branch(t, K, mode)


def prm_sync_status(ctx, stream: int = 0) -> int:
    return load().prm_sync_status(ctx, c_void_p(stream))


def prm_debug_last_direction(ctx, idx: int, host_out: int) -> None:
    """host_out: address of rows * cols writable host floats."""
    check(load().prm_debug_last_direction(ctx, idx, c_void_p(host_out)), "prm_debug_last_direction", ctx)


def prm_debug_withhold_tall_norms(ctx, stripe: int, wait_limit_s: float) -> None:
    check(load().prm_debug_withhold_tall_norms(ctx, stripe, wait_limit_s), "prm_debug_withhold_tall_norms", ctx)


def prm_profile(ctx, enable: bool) -> None:
    check(load().prm_profile(ctx, 1 if enable else 0), "prm_profile", ctx)


def prm_profile_read(ctx, family: int = -1):
    """(total_ms, records, kernels, work) for one kernel family or all (-1)."""
    ms, w = ctypes.c_double(), ctypes.c_double()
    n, k = c_int64(), c_int64()
    check(load().prm_profile_read(ctx, family, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(k), ctypes.byref(w)),
          "prm_profile_read", ctx)
    return ms.value, n.value, k.value, w.value


def prm_ns_gram(X: int, C: int, scale: int, gain: float, diag: float, out_dtype: int, batch: int, r: int, c: int,
                ldc: int, ldr: int, stream: int = 0):
    check(load().prm_ns_gram(c_void_p(X), c_void_p(C), c_void_p(scale), gain, diag, out_dtype, batch, r, c, ldc,
                             ldr, c_void_p(stream)), "prm_ns_gram")


def prm_ns_poly(C: int, P: int, gain: float, diag: float, in_dtype: int, batch: int, r: int, ldr: int,
                stream: int = 0):
    check(load().prm_ns_poly(c_void_p(C), c_void_p(P), gain, diag, in_dtype, batch, r, ldr, c_void_p(stream)),
          "prm_ns_poly")


def prm_ns_combine(X: int, P: int, Xout: int, scale: int, batch: int, r: int, c: int, ldc: int, ldr: int,
                   stream: int = 0):
    check(load().prm_ns_combine(c_void_p(X), c_void_p(P), c_void_p(Xout), c_void_p(scale), batch, r, c, ldc, ldr,
                                c_void_p(stream)), "prm_ns_combine")


def prm_rownorm_tall_step_noalloc(param: int, momentum: int, grad: int, grad_dtype: int, rows: int, cols: int,
                                  gamma: float, lr: float, wd: float, beta: float, eps: float,
                                  shape_scale: float = 0.0, stream: int = 0) -> None:
    check(load().prm_rownorm_tall_step_noalloc(c_void_p(param), c_void_p(momentum), c_void_p(grad), grad_dtype,
                                               rows, cols, gamma, lr, wd, beta, eps, shape_scale,
                                               c_void_p(stream)), "prm_rownorm_tall_step_noalloc")


def prm_adamw_step(param: int, exp_avg: int, exp_avg_sq: int, grad: int, grad_dtype: int, n: int, t: int,
                   lr: float, beta1: float, beta2: float, eps: float, wd: float, stream: int = 0) -> None:
    check(load().prm_adamw_step(c_void_p(param), c_void_p(exp_avg), c_void_p(exp_avg_sq), c_void_p(grad),
                                grad_dtype, n, t, lr, beta1, beta2, eps, wd, c_void_p(stream)), "prm_adamw_step")


def prm_newton_schulz_workspace(batch: int, m: int, n: int) -> int:
    out = c_size_t()
    check(load().prm_newton_schulz_workspace(batch, m, n, ctypes.byref(out)), "prm_newton_schulz_workspace")
    return out.value


def prm_newton_schulz(inp: int, out: int, batch: int, m: int, n: int, ns_coeffs, steps: int, ws: int,
                      ws_bytes: int, stream: int = 0):
    check(load().prm_newton_schulz(c_void_p(inp), c_void_p(out), batch, m, n, _coeff_ptr(ns_coeffs), steps,
                                   c_void_p(ws), ws_bytes, c_void_p(stream)), "prm_newton_schulz")
