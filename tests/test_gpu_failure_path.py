"""The failure path of the bounded waits, exercised without a fault (GPU).

The staged kernels wait on mbarriers for their bulk copies; every such wait
gives up after a time limit, records RN_DEVERR_STAGED_TIMEOUT in the device
error word and lets the kernel return. rn_selftest_bounded_wait runs that
same wait on a barrier nothing ever completes, with a short limit, so the
timeout branch runs for real; the test then checks that the host sees the
flag, that clearing it works, and that the context still runs a staged
normalization correctly.
"""
import numpy as np
import pytest

import gpu_util as G
import parity
import workloads
from oracle import reference
from row_wise_normalization_gb300 import capi

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    torch = G.torch_cuda()
    capi.device_error(clear=True)                          # start from a clean word
    assert capi.device_error(clear=False) == 0
    capi.check(capi.selftest_bounded_wait(20000, G.stream_handle()))   # 20 ms
    torch.cuda.synchronize()
    flags = capi.device_error(clear=True)
    assert flags & capi.RN_DEVERR_STAGED_TIMEOUT
    assert capi.device_error(clear=False) == 0
    # the context is still usable: a staged LayerNorm against the oracle
    wl = workloads.Workload("ln", 37, 20000, seed=901)
    x = wl.x()
    g, b = wl.params()
    y, m, r = G.run_ln(x, g, b, variant=capi.RN_VARIANT_STAGED)
    yr, mr, sr = reference.layer_norm(x, g, b)
    parity.check_y(y, yr)
    parity.check_rstd(r, sr)
    assert capi.device_error(clear=False) == 0
