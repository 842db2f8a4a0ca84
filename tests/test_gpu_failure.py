"""Failure detection on the GPU without a fault: a pipeline wait that can never
complete gives up after its limit, the status word records it, and the context
stays usable for correct work afterwards."""
import time

import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import assert_dual_equal, require_gpu, run_dual

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_bounded_wait_runs_out_and_reports():
    mxq.device_status(clear=True)
    t0 = time.perf_counter()
    mxq.selftest_wait_timeout(50_000_000)          # 50 ms, nothing ever arrives
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert 0.04 <= dt < 3.0, dt
    assert mxq.device_status(clear=True) & mxq.DEV_TIMEOUT
    assert mxq.device_status(clear=True) == 0       # cleared
    # the context is intact: a real launch afterwards is still byte-exact
    x, offs = W.dual_small()
    assert_dual_equal(run_dual(x, offs), oracle.mxfp8_dual(x, offs))
    assert mxq.device_status(clear=True) == 0


def test_selftest_limit_is_checked_on_the_host():
    with pytest.raises(mxq.MxqError) as e:
        mxq.selftest_wait_timeout(10)
    assert e.value.code == mxq.EBADSHAPE
