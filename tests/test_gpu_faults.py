"""Failure detection on the GPU without a GPU fault.

`inject_fault = 1` makes the producers issue nothing, so the MMA thread's
bounded wait on the first stage runs out (a barrier nothing signals).  The
kernel records the site in the device status word, every role leaves its loop,
tensor memory is freed, and tgemm_device_status reports
TGEMM_ERR_DEVICE_TIMEOUT.  The context must stay usable: a normal product
right after must be correct.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    H.tg()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("opts", [{"cta_group": 1}, {"cta_group": 2, "swap_ab": 1}, {"swap_ab": 2}, {"kernel": 2},
                                  {"kernel": 2, "cta_group": 2}],
                         ids=["one_sm", "cta_pair", "pair_swapped", "copy_producer", "copy_pair"])
def test_bounded_wait_reports_timeout_and_context_survives(opts):
    lib = H.tg()
    M, N, K = 512, 512, 256
    w = wl.Workload("fault", M, N, K, wl.BF16, "uniform", 60)
    A, B = wl.make_inputs(w)
    res = H.run_gpu(A, B, M, N, K, wl.BF16, check_status=False,
                    options={**opts, "inject_fault": 1, "wait_timeout_us": 200000})
    launch_status, device_status = res.status
    assert launch_status == lib.OK
    assert device_status == lib.ERR_DEVICE_TIMEOUT
    assert res.guard_ok and res.pad_ok
    # the status word was cleared and the context still computes correctly
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.device_status(stream) == lib.OK
    ok = H.run_gpu(A, B, M, N, K, wl.BF16, options={k: v for k, v in opts.items()})
    H.check_full(ok, A, B, M, N, K, wl.BF16, f"after fault {opts}")
