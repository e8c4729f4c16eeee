"""Build and call the plain-C float64 oracle (test infrastructure only).

``build()`` compiles ``rownorm_oracle.c`` with the host C compiler into a
shared library next to it; ``layer_norm`` / ``rms_norm`` call it through
ctypes with the same signatures and results as ``oracle.reference``.
Compiled with ``-ffp-contract=off`` and without fast-math so that the C
rounding order is the one written in the source on every host.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rownorm_oracle.c")
_LIB = os.path.join(_HERE, "librownorm_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle if its library is missing or older than the source."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call([cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_layer_norm.argtypes = [f, f, f, i64, i64, ctypes.c_float, f, f, f]
        lib.oracle_layer_norm.restype = None
        lib.oracle_rms_norm.argtypes = [f, f, i64, i64, ctypes.c_float, f, f]
        lib.oracle_rms_norm.restype = None
        _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def layer_norm(x, gamma, beta, eps=1e-5):
    """Same contract as ``oracle.reference.layer_norm``, computed in C."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    b = np.ascontiguousarray(beta, dtype=np.float32)
    rows, d = x.shape
    if d == 0:
        raise ValueError("d must be positive")
    y = np.empty((rows, d), np.float64)
    mean = np.empty(rows, np.float64)
    rstd = np.empty(rows, np.float64)
    lib.oracle_layer_norm(_p(x), _p(g), _p(b), rows, d, float(np.float32(eps)),
                          _p(y), _p(mean), _p(rstd))
    return y, mean, rstd


def rms_norm(x, w, eps=1e-5):
    """Same contract as ``oracle.reference.rms_norm``, computed in C."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, d = x.shape
    if d == 0:
        raise ValueError("d must be positive")
    y = np.empty((rows, d), np.float64)
    r = np.empty(rows, np.float64)
    lib.oracle_rms_norm(_p(x), _p(w), rows, d, float(np.float32(eps)), _p(y), _p(r))
    return y, r
