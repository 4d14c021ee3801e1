"""ctypes binding of ``include/kfac.h`` with the same names.

Argument marshalling only: every step of the computation runs in the CUDA
library.  Loading fails loudly when the library has not been built; there is
no fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os

__all__ = [
    "KFAC_OK", "KFAC_ERR_INVALID_ARG", "KFAC_ERR_NOT_SPD", "KFAC_ERR_CUDA",
    "KFAC_ERR_UNSUPPORTED", "KFAC_ERR_TIMEOUT", "KFAC_ERR_WORKSPACE",
    "KFAC_BF16", "KFAC_FP32", "KFAC_REFINE_NONE", "KFAC_REFINE_AUTO", "KFAC_REFINE_ALWAYS",
    "KFAC_PRECOND_FP32", "KFAC_PRECOND_AUTO",
    "kfac_factor_args", "kfac_running_args", "kfac_inverse_args", "kfac_precond_args",
    "KFACError", "lib", "library_path", "exported_symbols", "KERNEL_KINDS",
    "kfac_status_string", "kfac_version", "kfac_launch_count", "kfac_device_status", "kfac_wait_selftest",
    "kfac_profile", "kfac_profile_read", "kfac_profile_count", "kfac_profile_launch", "kfac_profile_timeline",
    "kfac_factors", "kfac_conv_factor_args", "kfac_conv_factors", "kfac_spatial_sum", "kfac_update_running",
    "kfac_damped_inverse_workspace", "kfac_damped_inverse",
    "kfac_precondition_workspace", "kfac_precondition", "kfac_precondition_static_capacity",
    "kfac_precondition_static", "kfac_pack_args", "kfac_pack_upper", "kfac_unpack_upper", "kfac_factor_tile_map",
]

KFAC_OK, KFAC_ERR_INVALID_ARG, KFAC_ERR_NOT_SPD, KFAC_ERR_CUDA = 0, 1, 2, 3
KFAC_ERR_UNSUPPORTED, KFAC_ERR_TIMEOUT, KFAC_ERR_WORKSPACE = 4, 5, 6
KFAC_BF16, KFAC_FP32 = 0, 1
KFAC_REFINE_NONE, KFAC_REFINE_AUTO, KFAC_REFINE_ALWAYS = 0, 1, 2
KFAC_PRECOND_FP32, KFAC_PRECOND_AUTO = 0, 1
KERNEL_KINDS = ("syrk", "running", "inv_panel", "inv_update", "inv_lauum", "gemm16", "gemm24", "conv_syrk",
                "inv_diag", "inv_prep", "inv_aux", "inv_newton")

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libkfac_gb300.so")


class kfac_factor_args(C.Structure):
    _fields_ = [("x", C.c_void_p), ("rows", C.c_int64), ("d", C.c_int64), ("ld_x", C.c_int64),
                ("out", C.c_void_p), ("ld_out", C.c_int64), ("stride_out", C.c_int64), ("scale", C.c_float)]


class kfac_conv_factor_args(C.Structure):
    _fields_ = [("x", C.c_void_p), ("B", C.c_int64), ("H", C.c_int64), ("W", C.c_int64), ("C", C.c_int64),
                ("out", C.c_void_p), ("ld_out", C.c_int64), ("stride_out", C.c_int64), ("scale", C.c_float)]


class kfac_running_args(C.Structure):
    _fields_ = [("shards", C.c_void_p), ("stride_shard", C.c_int64), ("running", C.c_void_p),
                ("damped", C.c_void_p), ("d", C.c_int64), ("ld", C.c_int64)]


class kfac_inverse_args(C.Structure):
    _fields_ = [("damped", C.c_void_p), ("inv", C.c_void_p), ("d", C.c_int64), ("ld_in", C.c_int64),
                ("ld_out", C.c_int64)]


class kfac_precond_args(C.Structure):
    _fields_ = [("inv_g", C.c_void_p), ("ld_g", C.c_int64), ("grad", C.c_void_p), ("ld_grad", C.c_int64),
                ("inv_a", C.c_void_p), ("ld_a", C.c_int64), ("out", C.c_void_p), ("ld_out", C.c_int64),
                ("d_out", C.c_int64), ("d_in", C.c_int64),
                ("weight", C.c_void_p), ("ld_weight", C.c_int64), ("lr", C.c_float)]


class kfac_pack_args(C.Structure):
    _fields_ = [("mat", C.c_void_p), ("d", C.c_int64), ("ld", C.c_int64), ("packed", C.c_void_p)]


exported_symbols = (
    "kfac_status_string", "kfac_version", "kfac_launch_count", "kfac_device_status", "kfac_wait_selftest",
    "kfac_profile", "kfac_profile_read", "kfac_profile_count", "kfac_profile_launch", "kfac_factors",
    "kfac_conv_factors", "kfac_spatial_sum",
    "kfac_update_running", "kfac_damped_inverse_workspace", "kfac_damped_inverse",
    "kfac_precondition_workspace", "kfac_precondition", "kfac_precondition_static_capacity",
    "kfac_precondition_static", "kfac_pack_upper", "kfac_unpack_upper", "kfac_factor_tile_map",
)

_lib = None


def lib() -> C.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise ImportError(
            f"K-FAC CUDA library not found at {library_path}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    L = C.CDLL(library_path)
    P = C.POINTER
    sig = {
        "kfac_status_string": (C.c_char_p, [C.c_int]),
        "kfac_version": (C.c_int, []),
        "kfac_launch_count": (C.c_ulonglong, []),
        "kfac_device_status": (C.c_int, [P(C.c_int), C.c_int, C.c_void_p]),
        "kfac_wait_selftest": (C.c_int, [C.c_int64, C.c_void_p]),
        "kfac_profile": (C.c_int, [C.c_int]),
        "kfac_profile_read": (C.c_int, [C.c_int, P(C.c_int64), P(C.c_double), P(C.c_double)]),
        "kfac_profile_count": (C.c_int, [P(C.c_int64)]),
        "kfac_profile_launch": (C.c_int, [C.c_int64, P(C.c_int), P(C.c_double), P(C.c_double), P(C.c_double)]),
        "kfac_factors": (C.c_int, [C.c_int, P(kfac_factor_args), C.c_int, C.c_int, C.c_int, C.c_void_p]),
        "kfac_conv_factors": (C.c_int, [C.c_int, P(kfac_conv_factor_args), C.c_int, C.c_int, C.c_void_p]),
        "kfac_spatial_sum": (C.c_int, [C.c_void_p, C.c_int, C.c_int64, C.c_int64, C.c_int64, C.c_int64,
                                       C.c_void_p, C.c_int64, C.c_void_p]),
        "kfac_update_running": (C.c_int, [C.c_int, P(kfac_running_args), C.c_int, C.c_float, C.c_float,
                                          C.c_int, C.c_void_p]),
        "kfac_damped_inverse_workspace": (C.c_size_t, [C.c_int, P(kfac_inverse_args), C.c_int]),
        "kfac_damped_inverse": (C.c_int, [C.c_int, P(kfac_inverse_args), C.c_float, C.c_int, C.c_void_p,
                                          C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
        "kfac_precondition_workspace": (C.c_size_t, [C.c_int, P(kfac_precond_args)]),
        "kfac_precondition": (C.c_int, [C.c_int, P(kfac_precond_args), C.c_int, C.c_void_p, C.c_void_p, C.c_size_t,
                                        C.c_void_p]),
        "kfac_precondition_static_capacity": (C.c_size_t, []),
        "kfac_precondition_static": (C.c_int, [C.c_int, P(kfac_precond_args), C.c_int, C.c_void_p, C.c_void_p]),
        "kfac_pack_upper": (C.c_int, [C.c_int, P(kfac_pack_args), C.c_void_p]),
        "kfac_unpack_upper": (C.c_int, [C.c_int, P(kfac_pack_args), C.c_int, C.c_void_p]),
        "kfac_factor_tile_map": (C.c_int, [C.c_int64, C.c_int64, P(C.c_int32), P(C.c_int64), P(C.c_int32),
                                           P(C.c_int64)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


class KFACError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {kfac_status_string(status)} ({status})")


def _check(fn: str, status: int) -> int:
    if status != KFAC_OK:
        raise KFACError(fn, status)
    return status


def _arr(struct, items):
    n = len(items)
    a = (struct * max(n, 1))(*items)
    return n, a


def kfac_status_string(status: int) -> str:
    return lib().kfac_status_string(status).decode()


def kfac_version() -> int:
    return lib().kfac_version()


def kfac_launch_count() -> int:
    return int(lib().kfac_launch_count())


def kfac_device_status(clear: bool = False, stream: int = 0) -> int:
    v = C.c_int(0)
    _check("kfac_device_status", lib().kfac_device_status(C.byref(v), int(clear), stream))
    return v.value


def kfac_wait_selftest(limit_cycles: int, stream: int = 0, check: bool = True) -> int:
    """One CTA's bounded wait on an mbarrier nothing arrives on (records KFAC_ERR_TIMEOUT)."""
    st = lib().kfac_wait_selftest(int(limit_cycles), stream)
    return _check("kfac_wait_selftest", st) if check else st


def kfac_profile(enable: bool) -> None:
    """Start (clearing the record) or stop the per-launch timing of the main kernels."""
    _check("kfac_profile", lib().kfac_profile(int(bool(enable))))


def kfac_profile_read(kind) -> dict:
    """Launches, summed duration (ms) and summed work of one kernel kind (a name of
    KERNEL_KINDS or its index); synchronises on the recorded events."""
    k = KERNEL_KINDS.index(kind) if isinstance(kind, str) else int(kind)
    n, ms, w = C.c_int64(0), C.c_double(0.0), C.c_double(0.0)
    _check("kfac_profile_read", lib().kfac_profile_read(k, C.byref(n), C.byref(ms), C.byref(w)))
    return {"launches": int(n.value), "ms": float(ms.value), "work": float(w.value)}


def kfac_profile_count() -> int:
    n = C.c_int64(0)
    _check("kfac_profile_count", lib().kfac_profile_count(C.byref(n)))
    return int(n.value)


def kfac_profile_launch(i: int) -> dict:
    """The i-th recorded launch: kind name, start and end (ms on a common axis), work."""
    k, a, b, w = C.c_int(0), C.c_double(0.0), C.c_double(0.0), C.c_double(0.0)
    _check("kfac_profile_launch", lib().kfac_profile_launch(i, C.byref(k), C.byref(a), C.byref(b), C.byref(w)))
    return {"kind": KERNEL_KINDS[k.value], "start_ms": float(a.value), "end_ms": float(b.value),
            "work": float(w.value)}


def kfac_profile_timeline() -> list:
    """Every recorded launch, in issue order."""
    return [kfac_profile_launch(i) for i in range(kfac_profile_count())]


def kfac_factors(args, dtype: int, P: int, mirror: int = 0, stream: int = 0, check: bool = True) -> int:
    n, a = _arr(kfac_factor_args, args)
    st = lib().kfac_factors(n, a, dtype, P, mirror, stream)
    return _check("kfac_factors", st) if check else st


def kfac_conv_factors(args, P: int, mirror: int = 0, stream: int = 0, check: bool = True) -> int:
    """Conv factors straight from NHWC bf16 activations (implicit im2col)."""
    n, a = _arr(kfac_conv_factor_args, args)
    st = lib().kfac_conv_factors(n, a, P, mirror, stream)
    return _check("kfac_conv_factors", st) if check else st


def kfac_spatial_sum(g: int, dtype: int, batch: int, hw: int, C_: int, ld_g: int, gs: int, ld_gs: int,
                     stream: int = 0, check: bool = True) -> int:
    st = lib().kfac_spatial_sum(g, dtype, batch, hw, C_, ld_g, gs, ld_gs, stream)
    return _check("kfac_spatial_sum", st) if check else st


def kfac_update_running(args, P: int, decay: float, gamma: float, first_step: bool, stream: int = 0,
                        check: bool = True) -> int:
    n, a = _arr(kfac_running_args, args)
    st = lib().kfac_update_running(n, a, P, decay, gamma, int(first_step), stream)
    return _check("kfac_update_running", st) if check else st


def kfac_damped_inverse_workspace(args, refine: int) -> int:
    n, a = _arr(kfac_inverse_args, args)
    return lib().kfac_damped_inverse_workspace(n, a, refine)


def kfac_damped_inverse(args, gamma_extra: float, refine: int, info: int, route: int, workspace: int,
                        workspace_bytes: int, stream: int = 0, check: bool = True) -> int:
    n, a = _arr(kfac_inverse_args, args)
    st = lib().kfac_damped_inverse(n, a, gamma_extra, refine, info, route, workspace, workspace_bytes, stream)
    return _check("kfac_damped_inverse", st) if check else st


def kfac_precondition_workspace(args) -> int:
    n, a = _arr(kfac_precond_args, args)
    return lib().kfac_precondition_workspace(n, a)


def kfac_precondition(args, precision: int, route: int, workspace: int, workspace_bytes: int, stream: int = 0,
                      check: bool = True) -> int:
    n, a = _arr(kfac_precond_args, args)
    st = lib().kfac_precondition(n, a, precision, route, workspace, workspace_bytes, stream)
    return _check("kfac_precondition", st) if check else st


def kfac_precondition_static_capacity() -> int:
    return int(lib().kfac_precondition_static_capacity())


def kfac_precondition_static(args, precision: int, route: int, stream: int = 0, check: bool = True) -> int:
    """kfac_precondition with the library's own fixed scratch (no workspace, no allocation)."""
    n, a = _arr(kfac_precond_args, args)
    st = lib().kfac_precondition_static(n, a, precision, route, stream)
    return _check("kfac_precondition_static", st) if check else st


def kfac_pack_upper(args, stream: int = 0, check: bool = True) -> int:
    """Packed upper triangles of every matrix of `args`, one launch."""
    n, a = _arr(kfac_pack_args, args)
    st = lib().kfac_pack_upper(n, a, stream)
    return _check("kfac_pack_upper", st) if check else st


def kfac_unpack_upper(args, mirror: bool = False, stream: int = 0, check: bool = True) -> int:
    """Upper triangles (with `mirror` the full symmetric matrices) from packed ones, one launch."""
    n, a = _arr(kfac_pack_args, args)
    st = lib().kfac_unpack_upper(n, a, int(bool(mirror)), stream)
    return _check("kfac_unpack_upper", st) if check else st


def kfac_factor_tile_map(d: int):
    """The (row_block, col_start, width) work units of a d x d factor."""
    cnt = C.c_int64(0)
    _check("kfac_factor_tile_map", lib().kfac_factor_tile_map(d, 0, None, None, None, C.byref(cnt)))
    n = cnt.value
    rb = (C.c_int32 * n)()
    cs = (C.c_int64 * n)()
    w = (C.c_int32 * n)()
    _check("kfac_factor_tile_map", lib().kfac_factor_tile_map(d, n, rb, cs, w, C.byref(cnt)))
    return [(rb[i], cs[i], w[i]) for i in range(n)]
