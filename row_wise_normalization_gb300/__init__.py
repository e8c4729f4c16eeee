"""Row-wise LayerNorm / RMSNorm forward on GB300 (sm_103a).

A thin torch-facing binding over the C ABI of ``librownorm.so``
(include/rownorm.h): it checks tensor shapes and dtypes, allocates outputs
with torch when the caller does not pass them, and hands raw device pointers
and the current CUDA stream to the library. Every arithmetic step runs in the
library's CUDA kernels; if the library is missing, calls raise.
"""
from __future__ import annotations

from . import capi
from .capi import RowNormError, load  # noqa: F401

__all__ = ["ln_fwd", "rms_fwd", "ln_fwd_residual", "rms_fwd_residual", "ln_fwd_batched",
           "rms_fwd_batched", "ln_bwd", "rms_bwd", "capi", "RowNormError", "load"]


def _stream_handle(t, stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(t.device if t.is_cuda else None)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _empty_like_home(x, shape, dtype=None):
    import torch

    dtype = torch.float32 if dtype is None else dtype
    if x.is_cuda:
        return torch.empty(shape, dtype=dtype, device=x.device)
    return torch.empty(shape, dtype=dtype, pin_memory=x.is_pinned())


_PAGEABLE = {}


def _pageable_ok():
    """Whether the current GPU reads pageable host memory (asked once per
    device)."""
    import torch

    if not torch.cuda.is_available():
        return False
    dev = torch.cuda.current_device()
    if dev not in _PAGEABLE:
        _PAGEABLE[dev] = capi.pageable_host_access()
    return _PAGEABLE[dev]


def _dtype_code(t):
    import torch

    codes = {torch.float32: capi.RN_DTYPE_F32, torch.bfloat16: capi.RN_DTYPE_BF16,
             torch.float16: capi.RN_DTYPE_F16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype} (float32, bfloat16 or float16)")
    return codes[t.dtype]


def _check_f32_cuda(name, t, dtype=None, contiguous=True):
    """Contiguous, of the expected dtype (FP32 unless given), and addressable
    by the GPU: a CUDA tensor, a pinned CPU tensor, or, on a GPU that reads
    pageable host memory (GB300), any CPU tensor (the kernel reads or writes
    host tensors over the host link)."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or t.is_pinned() or (t.device.type == "cpu" and _pageable_ok())):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned CPU tensor (this GPU "
                         f"does not read pageable host memory)")
    want = torch.float32 if dtype is None else dtype
    if t.dtype != want:
        raise TypeError(f"{name} must be {want}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _rows_of(name, t, d):
    """(rows, row stride) of x or y: a contiguous tensor of rows of d, or a
    2-D tensor whose rows are d contiguous elements at a stride >= d (a column
    block of a wider matrix)."""
    if t.is_contiguous():
        return (t.numel() // d if d else 0), d
    if t.dim() == 2 and t.shape[1] == d and t.stride(1) == 1 and t.stride(0) >= d:
        return t.shape[0], t.stride(0)
    raise ValueError(f"{name} must be contiguous, or 2-D with unit column stride and a row "
                     f"stride >= its width")


def ln_fwd(x, gamma, beta, eps: float = 1e-5, *, y=None, mean=None, rstd=None, stream=None,
           variant: int = capi.RN_VARIANT_AUTO):
    """LayerNorm forward over the last dimension of ``x``.

    x, gamma, beta (and y) are float32, bfloat16 or float16 -- all the same
    type; statistics are computed in FP32. Returns ``(y, mean, rstd)``: y like
    x; mean and rstd FP32 of shape x.shape[:-1]. Tensors are CUDA tensors or
    pinned CPU tensors, or any CPU tensors on a GPU that reads pageable host
    memory (read or written by the kernel over the host link);
    outputs not passed in are allocated where x lives. x and y may also be
    2-D row-strided views (``big[:, a:a + d]``): the kernels then read and
    write the rows in place.
    """
    code = _dtype_code(x)
    _check_f32_cuda("x", x, x.dtype, contiguous=False)
    d = x.shape[-1]
    rows, ldx = _rows_of("x", x, d)
    for n, t in (("gamma", gamma), ("beta", beta)):
        _check_f32_cuda(n, t, x.dtype)
        if t.numel() != d:
            raise ValueError(f"{n} must have {d} elements")
    if y is None:
        y = _empty_like_home(x, x.shape, x.dtype)
    if mean is None:
        mean = _empty_like_home(x, x.shape[:-1])
    if rstd is None:
        rstd = _empty_like_home(x, x.shape[:-1])
    _check_f32_cuda("y", y, x.dtype, contiguous=False)
    if y.numel() != x.numel() or y.shape[-1] != d:
        raise ValueError("y must be shaped like x")
    _, ldy = _rows_of("y", y, d)
    for n, t in (("mean", mean), ("rstd", rstd)):
        _check_f32_cuda(n, t)
        if t.numel() != rows:
            raise ValueError(f"{n} must have {rows} elements")
    if ldx == d and ldy == d:
        st = capi.ln_fwd_typed(code, variant, x.data_ptr(), gamma.data_ptr(), beta.data_ptr(),
                               y.data_ptr(), mean.data_ptr(), rstd.data_ptr(), rows, d,
                               float(eps), _stream_handle(x, stream))
    else:
        st = capi.ln_fwd_strided(code, variant, x.data_ptr(), ldx, gamma.data_ptr(),
                                 beta.data_ptr(), y.data_ptr(), ldy, mean.data_ptr(),
                                 rstd.data_ptr(), rows, d, float(eps), _stream_handle(x, stream))
    capi.check(st)
    return y, mean, rstd


def rms_fwd(x, w, eps: float = 1e-5, *, y=None, stream=None,
            variant: int = capi.RN_VARIANT_AUTO):
    """RMSNorm forward over the last dimension of ``x`` (float32, bfloat16 or
    float16; w of the same type); returns y. x and y may be 2-D row-strided
    views, as in ln_fwd."""
    code = _dtype_code(x)
    _check_f32_cuda("x", x, x.dtype, contiguous=False)
    d = x.shape[-1]
    rows, ldx = _rows_of("x", x, d)
    _check_f32_cuda("w", w, x.dtype)
    if w.numel() != d:
        raise ValueError(f"w must have {d} elements")
    if y is None:
        y = _empty_like_home(x, x.shape, x.dtype)
    _check_f32_cuda("y", y, x.dtype, contiguous=False)
    if y.numel() != x.numel() or y.shape[-1] != d:
        raise ValueError("y must be shaped like x")
    _, ldy = _rows_of("y", y, d)
    if ldx == d and ldy == d:
        st = capi.rms_fwd_typed(code, variant, x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, d,
                                float(eps), _stream_handle(x, stream))
    else:
        st = capi.rms_fwd_strided(code, variant, x.data_ptr(), ldx, w.data_ptr(), y.data_ptr(),
                                  ldy, rows, d, float(eps), _stream_handle(x, stream))
    capi.check(st)
    return y


def _batched(op, problems, eps, stream):
    if not problems:
        return []
    x0 = problems[0][0]
    code = _dtype_code(x0)
    items, outs = [], []
    for k, pr in enumerate(problems):
        x, params = pr[0], pr[1:]
        _check_f32_cuda(f"problem {k} x", x, x0.dtype)
        d = x.shape[-1]
        rows = x.numel() // d if d else 0
        for t in params:
            _check_f32_cuda(f"problem {k} parameter", t, x0.dtype)
            if t.numel() != d:
                raise ValueError(f"problem {k}: parameters must have {d} elements")
        y = _empty_like_home(x, x.shape, x.dtype)
        if op == capi.RN_OP_LN:
            mean = _empty_like_home(x, x.shape[:-1])
            rstd = _empty_like_home(x, x.shape[:-1])
            items.append((x.data_ptr(), params[0].data_ptr(), params[1].data_ptr(), y.data_ptr(),
                          mean.data_ptr(), rstd.data_ptr(), rows, d))
            outs.append((y, mean, rstd))
        else:
            items.append((x.data_ptr(), params[0].data_ptr(), 0, y.data_ptr(), 0, 0, rows, d))
            outs.append(y)
    fn = capi.ln_fwd_batched if op == capi.RN_OP_LN else capi.rms_fwd_batched
    capi.check(fn(code, capi.problems(items), len(items), float(eps), _stream_handle(x0, stream)))
    return outs


def ln_fwd_batched(problems, eps: float = 1e-5, *, stream=None):
    """LayerNorm of many small tensors in as few launches as possible.

    ``problems``: a sequence of ``(x, gamma, beta)``, contiguous, all of one
    dtype (float32, bfloat16 or float16). Returns a list of ``(y, mean,
    rstd)``, one per problem. Problems of width <= 1024 share one launch per
    128; wider ones get their own.
    """
    return _batched(capi.RN_OP_LN, problems, eps, stream)


def rms_fwd_batched(problems, eps: float = 1e-5, *, stream=None):
    """RMSNorm of many small tensors: ``problems`` is a sequence of ``(x, w)``;
    returns the list of y."""
    return _batched(capi.RN_OP_RMS, problems, eps, stream)


def _check_like(name, t, numel):
    _check_f32_cuda(name, t)
    if t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements")


def ln_fwd_residual(x, res, gamma, beta, eps: float = 1e-5, *, h=None, y=None, mean=None,
                    rstd=None, write_h: bool = True, stream=None,
                    variant: int = capi.RN_VARIANT_AUTO):
    """h = x + res, then LayerNorm of h over the last dimension, in one kernel.

    Returns ``(h, y, mean, rstd)``; h is None when ``write_h`` is False and no
    h tensor is passed. Tensors are CUDA tensors or host tensors as for ln_fwd.
    """
    _check_f32_cuda("x", x)
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    _check_like("res", res, x.numel())
    _check_like("gamma", gamma, d)
    _check_like("beta", beta, d)
    if h is None and write_h:
        h = _empty_like_home(x, x.shape)
    y = _empty_like_home(x, x.shape) if y is None else y
    mean = _empty_like_home(x, x.shape[:-1]) if mean is None else mean
    rstd = _empty_like_home(x, x.shape[:-1]) if rstd is None else rstd
    if h is not None:
        _check_like("h", h, x.numel())
    _check_like("y", y, x.numel())
    _check_like("mean", mean, rows)
    _check_like("rstd", rstd, rows)
    st = capi.ln_fwd_residual_variant(variant, x.data_ptr(), res.data_ptr(), gamma.data_ptr(),
                                      beta.data_ptr(), h.data_ptr() if h is not None else 0,
                                      y.data_ptr(), mean.data_ptr(), rstd.data_ptr(), rows, d,
                                      float(eps), _stream_handle(x, stream))
    capi.check(st)
    return h, y, mean, rstd


def rms_fwd_residual(x, res, w, eps: float = 1e-5, *, h=None, y=None, write_h: bool = True,
                     stream=None, variant: int = capi.RN_VARIANT_AUTO):
    """h = x + res, then RMSNorm of h over the last dimension, in one kernel.

    Returns ``(h, y)``; h is None when ``write_h`` is False and none is passed.
    """
    _check_f32_cuda("x", x)
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    _check_like("res", res, x.numel())
    _check_like("w", w, d)
    if h is None and write_h:
        h = _empty_like_home(x, x.shape)
    y = _empty_like_home(x, x.shape) if y is None else y
    if h is not None:
        _check_like("h", h, x.numel())
    _check_like("y", y, x.numel())
    st = capi.rms_fwd_residual_variant(variant, x.data_ptr(), res.data_ptr(), w.data_ptr(),
                                       h.data_ptr() if h is not None else 0, y.data_ptr(), rows,
                                       d, float(eps), _stream_handle(x, stream))
    capi.check(st)
    return h, y


def _workspace(op, rows, d, device, workspace):
    import torch

    if workspace is not None:
        return workspace
    nbytes = capi.bwd_workspace_size(op, rows, d)
    return torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=device)


def ln_bwd(dy, x, gamma, mean, rstd, *, dx=None, dgamma=None, dbeta=None,
           param_grads: bool = True, workspace=None, stream=None):
    """LayerNorm backward from the forward's saved mean and rstd. dy, x and
    gamma are float32, bfloat16 or float16 (one type; dx and the parameter
    gradients come back in it); mean and rstd are FP32. Returns ``(dx,
    dgamma, dbeta)`` (the last two None when ``param_grads`` is False).
    ``workspace``: a float32 CUDA tensor for the parameter-gradient partials
    (allocated if not given)."""
    import torch

    code = _dtype_code(x)
    for n, t in (("dy", dy), ("x", x), ("gamma", gamma)):
        _check_f32_cuda(n, t, x.dtype)
    for n, t in (("mean", mean), ("rstd", rstd)):
        _check_f32_cuda(n, t)
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    dx = torch.empty_like(x) if dx is None else dx
    if param_grads:
        dgamma = torch.empty(d, dtype=x.dtype, device=x.device) if dgamma is None else dgamma
        dbeta = torch.empty(d, dtype=x.dtype, device=x.device) if dbeta is None else dbeta
        ws = _workspace(capi.RN_OP_LN, rows, d, x.device, workspace)
    else:
        dgamma = dbeta = ws = None
    st = capi.ln_bwd_typed(code, dy.data_ptr(), x.data_ptr(), gamma.data_ptr(), mean.data_ptr(),
                           rstd.data_ptr(), dx.data_ptr(),
                           dgamma.data_ptr() if dgamma is not None else 0,
                           dbeta.data_ptr() if dbeta is not None else 0, rows, d,
                           ws.data_ptr() if ws is not None else 0,
                           ws.numel() * 4 if ws is not None else 0, _stream_handle(x, stream))
    capi.check(st)
    return dx, dgamma, dbeta


def rms_bwd(dy, x, w, eps: float = 1e-5, *, dx=None, dw=None, param_grads: bool = True,
            workspace=None, stream=None):
    """RMSNorm backward (float32, bfloat16 or float16 tensors of one type).
    Returns ``(dx, dw)``."""
    import torch

    code = _dtype_code(x)
    for n, t in (("dy", dy), ("x", x), ("w", w)):
        _check_f32_cuda(n, t, x.dtype)
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    dx = torch.empty_like(x) if dx is None else dx
    if param_grads:
        dw = torch.empty(d, dtype=x.dtype, device=x.device) if dw is None else dw
        ws = _workspace(capi.RN_OP_RMS, rows, d, x.device, workspace)
    else:
        dw = ws = None
    st = capi.rms_bwd_typed(code, dy.data_ptr(), x.data_ptr(), w.data_ptr(), dx.data_ptr(),
                            dw.data_ptr() if dw is not None else 0, rows, d, float(eps),
                            ws.data_ptr() if ws is not None else 0,
                            ws.numel() * 4 if ws is not None else 0, _stream_handle(x, stream))
    capi.check(st)
    return dx, dw
