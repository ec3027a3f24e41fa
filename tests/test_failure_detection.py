"""Failure detection without a GPU fault: every mbarrier wait in the kernels is bounded; when it
runs out (here on a barrier nothing arrives at) the kernel records XY_DEV_TIMEOUT and returns,
and the CUDA context stays usable for the next step."""

import numpy as np
import pytest
import torch

import workloads
from gpu_cases import assert_parity, run

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    xy.xy_selftest_bounded_wait(20000, err, res)      # a 20 ms limit
    torch.cuda.synchronize()
    timed_out_ok, waited_us, aborted_ok = res.cpu().tolist()
    assert timed_out_ok == 0 and aborted_ok == 0
    assert 20000 <= waited_us < 1000000
    assert int(err.item()) & 8                         # XY_DEV_TIMEOUT
    with pytest.raises(xy.XYDeviceError):
        xy.check_err_word(err)
    # the next step on the same context runs and matches the oracle
    assert_parity(run(workloads.tiny()))


def test_bounded_wait_rejects_bad_arguments():
    import paged_kv_varlen_xy_gb300 as xy
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.zeros(3, dtype=torch.int32, device="cuda")
    with pytest.raises(xy.XYError):
        xy.xy_selftest_bounded_wait(0, err, res)
