"""ctypes declarations of the C ABI in include/rownorm.h.

Argument marshalling only: every function here is the C entry point of
``librownorm.so`` with its argument and return types set. Pointers are plain
integers (device addresses), sizes are int64, eps is float32 and the stream
is a ``cudaStream_t`` passed as an integer (0 = legacy default stream).

Importing this module does not load the library; ``load()`` does, and fails
loudly if the library has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librownorm.so")

RN_OK = 0
RN_ERR_NULL = 1
RN_ERR_SIZE = 2
RN_ERR_EPS = 3
RN_ERR_ALIAS = 4
RN_ERR_CUDA = 5
RN_ERR_ALIGN = 6
RN_ERR_VARIANT = 7
RN_ERR_DTYPE = 8
RN_ERR_SCRATCH = 9
RN_ERR_HOSTMEM = 10

# device error word bits
RN_DEVERR_STAGED_TIMEOUT = 1
RN_DEVERR_CLUSTER_TIMEOUT = 2
RN_DEVERR_PARAMS_TIMEOUT = 4

# static scratch of ln_bwd_noalloc
RN_NOALLOC_SCRATCH_BYTES = 8 << 20
RN_NOALLOC_MAX_D = 4096

RN_DTYPE_F32 = 0
RN_DTYPE_BF16 = 1
RN_DTYPE_F16 = 2

RN_VARIANT_AUTO = 0
RN_VARIANT_WARP = 1
RN_VARIANT_BLOCK = 2
RN_VARIANT_STAGED = 3
RN_VARIANT_STREAM = 4
RN_VARIANT_CLUSTER = 5
RN_VARIANT_COUNT = 6

RN_OP_LN = 0
RN_OP_RMS = 1

# Every function include/rownorm.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_INT = ctypes.c_int


class rn_plan(ctypes.Structure):
    _fields_ = [("variant", _INT), ("vec", _INT), ("slots", _INT), ("threads_per_row", _INT),
                ("rows_per_cta", _INT), ("threads_per_cta", _INT), ("smem_bytes", _INT),
                ("prefetch", _INT), ("params_held", _INT), ("aligned", _INT),
                ("cluster", _INT)]


class rn_problem(ctypes.Structure):
    """One problem of ln_fwd_batched / rms_fwd_batched (pointers as ints)."""
    _fields_ = [("x", ctypes.c_void_p), ("p0", ctypes.c_void_p), ("p1", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("mean_out", ctypes.c_void_p),
                ("rstd_out", ctypes.c_void_p), ("rows", ctypes.c_int64), ("d", ctypes.c_int64)]


SIGNATURES = {
    "ln_fwd": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
    "rms_fwd": (_INT, [_P, _P, _P, _I64, _I64, _F, _P]),
    "rn_status_str": (ctypes.c_char_p, [_INT]),
    "rn_last_cuda_error": (_INT, []),
    "rn_plan_for": (_INT, [_INT, _INT, _I64, _P, _P, _P, _P, ctypes.POINTER(rn_plan)]),
    "rn_variant_name": (ctypes.c_char_p, [_INT]),
    "ln_fwd_variant": (_INT, [_INT, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
    "rms_fwd_variant": (_INT, [_INT, _P, _P, _P, _I64, _I64, _F, _P]),
    "rn_launch_empty": (_INT, [_I64, _INT, _P]),
    "ln_fwd_residual": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
    "rms_fwd_residual": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
    "ln_fwd_residual_variant": (_INT, [_INT, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
    "rms_fwd_residual_variant": (_INT, [_INT, _P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
    "rn_plan_for_residual": (_INT, [_INT, _INT, _I64, _P, _P, _P, _P, _P, _P,
                                    ctypes.POINTER(rn_plan)]),
    "ln_fwd_typed": (_INT, [_INT, _INT, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P]),
    "ln_bwd_workspace_size": (_INT, [_I64, _I64, ctypes.POINTER(ctypes.c_size_t)]),
    "rms_bwd_workspace_size": (_INT, [_I64, _I64, ctypes.POINTER(ctypes.c_size_t)]),
    "ln_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, ctypes.c_size_t, _P]),
    "rms_bwd": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
    "ln_bwd_noalloc": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P]),
    "ln_bwd_typed": (_INT, [_INT, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, ctypes.c_size_t,
                            _P]),
    "rms_bwd_typed": (_INT, [_INT, _P, _P, _P, _P, _P, _I64, _I64, _F, _P, ctypes.c_size_t, _P]),
    "rn_selftest_bounded_wait": (_INT, [ctypes.c_uint, _P]),
    "ln_fwd_batched": (_INT, [_INT, ctypes.POINTER(rn_problem), _INT, _F, _P]),
    "rms_fwd_batched": (_INT, [_INT, ctypes.POINTER(rn_problem), _INT, _F, _P]),
    "ln_fwd_strided": (_INT, [_INT, _INT, _P, _I64, _P, _P, _P, _I64, _P, _P, _I64, _I64, _F, _P]),
    "rms_fwd_strided": (_INT, [_INT, _INT, _P, _I64, _P, _P, _I64, _I64, _I64, _F, _P]),
    "rn_plan_for_strided": (_INT, [_INT, _INT, _INT, _I64, _P, _I64, _P, _I64, _P, _P,
                                   ctypes.POINTER(rn_plan)]),
    "rms_fwd_typed": (_INT, [_INT, _INT, _P, _P, _P, _I64, _I64, _F, _P]),
    "rn_plan_for_typed": (_INT, [_INT, _INT, _INT, _I64, _P, _P, _P, _P, ctypes.POINTER(rn_plan)]),
    "rn_device_error": (_INT, [ctypes.POINTER(ctypes.c_uint), _INT]),
    "rn_pageable_host_access": (_INT, [ctypes.POINTER(_INT)]),
}

_lib = None


class RowNormError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def load() -> ctypes.CDLL:
    """Load librownorm.so (once) and declare every entry point."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m row_wise_normalization_gb300.build` "
                "(or __graft_entry__.build()). There is no CPU fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_str(status: int) -> str:
    return load().rn_status_str(status).decode()


def check(status: int) -> None:
    """Raise RowNormError for a non-RN_OK status."""
    if status != RN_OK:
        msg = status_str(status)
        if status == RN_ERR_CUDA:
            msg += f" (cudaError {load().rn_last_cuda_error()})"
        raise RowNormError(status, msg)


def plan(op: int, variant: int, d: int, x: int, y: int, p0: int = 0, p1: int = 0) -> rn_plan:
    """The kernel configuration a call would launch (host only)."""
    out = rn_plan()
    check(load().rn_plan_for(op, variant, d, x, y, p0, p1, ctypes.byref(out)))
    return out


def plan_residual(op: int, variant: int, d: int, x: int, res: int, h: int, y: int, p0: int = 0,
                  p1: int = 0) -> rn_plan:
    """The kernel configuration a residual call would launch (host only)."""
    out = rn_plan()
    check(load().rn_plan_for_residual(op, variant, d, x, res, h, y, p0, p1, ctypes.byref(out)))
    return out


def plan_typed(dtype: int, op: int, variant: int, d: int, x: int, y: int, p0: int = 0,
               p1: int = 0) -> rn_plan:
    """The kernel configuration a typed call would launch (host only)."""
    out = rn_plan()
    check(load().rn_plan_for_typed(dtype, op, variant, d, x, y, p0, p1, ctypes.byref(out)))
    return out


def plan_strided(dtype: int, op: int, variant: int, d: int, x: int, ldx: int, y: int, ldy: int,
                 p0: int = 0, p1: int = 0) -> rn_plan:
    """The kernel configuration a strided call would launch (host only)."""
    out = rn_plan()
    check(load().rn_plan_for_strided(dtype, op, variant, d, x, ldx, y, ldy, p0, p1,
                                     ctypes.byref(out)))
    return out


def variant_name(v: int) -> str:
    return load().rn_variant_name(v).decode()


# Raw entry points (device pointers as ints), same names as the C ABI.
def ln_fwd(x, gamma, beta, y, mean_out, rstd_out, rows, d, eps, stream=0) -> int:
    return load().ln_fwd(x, gamma, beta, y, mean_out, rstd_out, rows, d, eps, stream)


def rms_fwd(x, w, y, rows, d, eps, stream=0) -> int:
    return load().rms_fwd(x, w, y, rows, d, eps, stream)


def ln_fwd_variant(variant, x, gamma, beta, y, mean_out, rstd_out, rows, d, eps, stream=0) -> int:
    return load().ln_fwd_variant(variant, x, gamma, beta, y, mean_out, rstd_out, rows, d, eps,
                                 stream)


def rms_fwd_variant(variant, x, w, y, rows, d, eps, stream=0) -> int:
    return load().rms_fwd_variant(variant, x, w, y, rows, d, eps, stream)


def launch_empty(grid, threads, stream=0) -> int:
    return load().rn_launch_empty(grid, threads, stream)


def pageable_host_access() -> bool:
    """Whether the current GPU reads pageable (unpinned) host memory."""
    out = ctypes.c_int(0)
    check(load().rn_pageable_host_access(ctypes.byref(out)))
    return out.value != 0


def device_error(clear: bool = False) -> int:
    """The device error word (0 when no kernel reported a problem)."""
    out = ctypes.c_uint(0)
    check(load().rn_device_error(ctypes.byref(out), 1 if clear else 0))
    return out.value


def ln_fwd_residual(x, res, gamma, beta, h_out, y, mean_out, rstd_out, rows, d, eps,
                    stream=0) -> int:
    return load().ln_fwd_residual(x, res, gamma, beta, h_out, y, mean_out, rstd_out, rows, d,
                                  eps, stream)


def rms_fwd_residual(x, res, w, h_out, y, rows, d, eps, stream=0) -> int:
    return load().rms_fwd_residual(x, res, w, h_out, y, rows, d, eps, stream)


def ln_fwd_residual_variant(variant, x, res, gamma, beta, h_out, y, mean_out, rstd_out, rows, d,
                            eps, stream=0) -> int:
    return load().ln_fwd_residual_variant(variant, x, res, gamma, beta, h_out, y, mean_out,
                                          rstd_out, rows, d, eps, stream)


def rms_fwd_residual_variant(variant, x, res, w, h_out, y, rows, d, eps, stream=0) -> int:
    return load().rms_fwd_residual_variant(variant, x, res, w, h_out, y, rows, d, eps, stream)


def ln_fwd_typed(dtype, variant, x, gamma, beta, y, mean_out, rstd_out, rows, d, eps,
                 stream=0) -> int:
    return load().ln_fwd_typed(dtype, variant, x, gamma, beta, y, mean_out, rstd_out, rows, d,
                               eps, stream)


def rms_fwd_typed(dtype, variant, x, w, y, rows, d, eps, stream=0) -> int:
    return load().rms_fwd_typed(dtype, variant, x, w, y, rows, d, eps, stream)


def bwd_workspace_size(op: int, rows: int, d: int) -> int:
    out = ctypes.c_size_t(0)
    fn = load().ln_bwd_workspace_size if op == RN_OP_LN else load().rms_bwd_workspace_size
    check(fn(rows, d, ctypes.byref(out)))
    return out.value


def ln_bwd(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, workspace, workspace_bytes,
           stream=0) -> int:
    return load().ln_bwd(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, workspace,
                         workspace_bytes, stream)


def rms_bwd(dy, x, w, dx, dw, rows, d, eps, workspace, workspace_bytes, stream=0) -> int:
    return load().rms_bwd(dy, x, w, dx, dw, rows, d, eps, workspace, workspace_bytes, stream)


def ln_bwd_noalloc(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, stream=0) -> int:
    """ln_bwd with its partials in the library's static scratch: for callers
    that cannot allocate device memory at that point (an allocator that holds
    nearly all of HBM, a loop that cannot take cudaFree's synchronisation).
    d <= RN_NOALLOC_MAX_D; calls that overlap on the GPU race on the scratch."""
    return load().ln_bwd_noalloc(dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, stream)


def ln_fwd_strided(dtype, variant, x, ldx, gamma, beta, y, ldy, mean, rstd, rows, d, eps,
                   stream=0) -> int:
    return load().ln_fwd_strided(dtype, variant, x, ldx, gamma, beta, y, ldy, mean, rstd, rows,
                                 d, eps, stream)


def rms_fwd_strided(dtype, variant, x, ldx, w, y, ldy, rows, d, eps, stream=0) -> int:
    return load().rms_fwd_strided(dtype, variant, x, ldx, w, y, ldy, rows, d, eps, stream)


def problems(items) -> "ctypes.Array":
    """A ctypes array of rn_problem from (x, p0, p1, y, mean, rstd, rows, d)
    tuples of ints."""
    arr = (rn_problem * max(len(items), 1))()
    for i, it in enumerate(items):
        arr[i] = rn_problem(*it)
    return arr


def ln_fwd_batched(dtype, probs, count, eps, stream=0) -> int:
    return load().ln_fwd_batched(dtype, probs, count, eps, stream)


def rms_fwd_batched(dtype, probs, count, eps, stream=0) -> int:
    return load().rms_fwd_batched(dtype, probs, count, eps, stream)


def selftest_bounded_wait(timeout_us: int, stream=0) -> int:
    """Launch the bounded-wait self-test (see include/rownorm.h)."""
    return load().rn_selftest_bounded_wait(timeout_us, stream)


def ln_bwd_typed(dtype, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d, workspace,
                 workspace_bytes, stream=0) -> int:
    return load().ln_bwd_typed(dtype, dy, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, d,
                               workspace, workspace_bytes, stream)


def rms_bwd_typed(dtype, dy, x, w, dx, dw, rows, d, eps, workspace, workspace_bytes,
                  stream=0) -> int:
    return load().rms_bwd_typed(dtype, dy, x, w, dx, dw, rows, d, eps, workspace,
                                workspace_bytes, stream)
