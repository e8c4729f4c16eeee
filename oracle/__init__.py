"""CPU oracle for row-wise LayerNorm and RMSNorm forward (float64).

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import, call, link or run anything in this package. The CUDA library never
does, and nothing here imports it: the two share no code.

Two independent restatements of the same definitions live here:

* ``reference`` -- NumPy, float64, vectorised over rows;
* ``rownorm_oracle.c`` -- plain C, float64, one row at a time (loaded through
  ``c_oracle``); this is the one timed as the CPU baseline.

Both take the exact FP32 inputs the GPU receives, widen them to float64 and
compute the plain definitions; both are pinned by ``tests/test_oracle_*.py``
(closed forms, invariants, exact brute force on tiny rows, a float64 library
cross-check and planted mistakes that the pins must catch).
"""
from .reference import (layer_norm, layer_norm_backward, layer_norm_residual,  # noqa: F401
                        residual_sum, rms_norm, rms_norm_backward, rms_norm_residual)
