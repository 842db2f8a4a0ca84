"""The no-allocation form of the three-pass cast.

mxq_quantize_2d_dual_3pass_noalloc exists for callers that cannot allocate
device memory when they need the cast (work recorded into a CUDA graph in
global capture mode, latency-critical paths where cudaMalloc/cudaFree may
synchronize the device, plugins under a framework allocator they cannot
reach); its workspace is a static device array inside the library.  Here it is
called through the C ABI and must give exactly the bytes of the workspace
form, mxq_quantize_2d_dual_3pass, on two calls in a row (the second with other
data, so nothing left in the shared array can leak into a result).  This file
is collected last so that a failure here never hides another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import FILL, assert_dual_equal, require_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu

MXQ_ESCRATCH = -8
SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _noalloc_entry():
    f = mxq.lib().mxq_quantize_2d_dual_3pass_noalloc
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int32, vp, vp, vp, vp, vp]
    return f


def _outputs(M, N):
    kw = dict(dtype=torch.uint8, device="cuda")
    return mxq.DualOutputs(torch.full((M, N), FILL, **kw), torch.full((M * N // 32,), FILL, **kw),
                           torch.full((N, M), FILL, **kw), torch.full((M * N // 32,), FILL, **kw))


def _bytes(out):
    return {k: getattr(out, k).cpu().numpy().reshape(-1) for k in out._fields}


def test_noalloc_matches_workspace_form_on_two_calls():
    f = _noalloc_entry()
    vp = ctypes.c_void_p
    cases = [(W.moe_grouped(M=4096, N=2048, experts=8, routed_units=28, seed=3), "moe"),
             ((W.dual_specials(2048, 1024, seed=4), np.array([0, 1024, 1024, 1920], np.int32)),
              "specials")]
    for (x_np, offs_np), tag in cases:
        M, N = x_np.shape
        x = to_dev_bf16(x_np)
        offs = torch.from_numpy(offs_np).cuda()
        got = _outputs(M, N)
        stream = torch.cuda.current_stream()
        rc = f(vp(x.data_ptr()), M, N, vp(offs.data_ptr()), offs.numel(),
               *(vp(t.data_ptr()) for t in got), vp(stream.cuda_stream))
        assert rc == mxq.OK, mxq.status_string(rc)
        ref = mxq.quantize_2d_dual_3pass(
            x, offs, workspace=torch.empty(M * N // 32, dtype=torch.uint8, device="cuda"),
            out=_outputs(M, N))
        torch.cuda.synchronize()
        assert_dual_equal(_bytes(got), _bytes(ref), f"{tag} ")


def test_noalloc_rejects_problems_beyond_its_scratch():
    f = _noalloc_entry()
    vp = ctypes.c_void_p
    M, N = 32768, 16512            # M*N/32 is just above 16 MiB
    assert M * N // 32 > SCRATCH_BYTES
    fake = [vp(1 << 20)] * 4       # never dereferenced: rejected on the host
    assert f(vp(1 << 20), M, N, None, 0, *fake, None) == MXQ_ESCRATCH
    assert "scratch" in mxq.status_string(MXQ_ESCRATCH)
