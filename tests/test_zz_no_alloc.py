"""The no-allocation form of the three-pass cast.

mxq_quantize_2d_dual_3pass_noalloc exists for callers that cannot allocate
device memory when they need the cast (work recorded into a CUDA graph in
global capture mode, latency-critical paths where cudaMalloc/cudaFree may
synchronize the device, plugins under a framework allocator they cannot
reach); its workspace is a static device array inside the library.  Here it is
called through the C ABI on several calls in a row (each with other data, so
nothing left in the shared array can leak into a result) and must give exactly
the oracle's bytes of the three-pass composition and the bytes of the
workspace form, mxq_quantize_2d_dual_3pass.  One tensor holds colwise blocks
with NaN, so the 32x1 pass's rule (NaN skipped by the amax) runs through the
static array.  A second test records the call into a CUDA graph in global
capture mode and replays it on fresh inputs.  This file is collected last so
that a failure here never hides another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import FILL, assert_dual_equal, require_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu

MXQ_ESCRATCH = -8
SCRATCH_BYTES = 16 << 20
VP = ctypes.c_void_p


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _noalloc_entry():
    f = mxq.lib().mxq_quantize_2d_dual_3pass_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [VP, ctypes.c_int64, ctypes.c_int64, VP, ctypes.c_int32, VP, VP, VP, VP, VP]
    return f


def _outputs(M, N):
    kw = dict(dtype=torch.uint8, device="cuda")
    return mxq.DualOutputs(torch.full((M, N), FILL, **kw), torch.full((M * N // 32,), FILL, **kw),
                           torch.full((N, M), FILL, **kw), torch.full((M * N // 32,), FILL, **kw))


def _bytes(out):
    return {k: getattr(out, k).cpu().numpy().reshape(-1) for k in out._fields}


def _call(f, x, offs, out, stream):
    M, N = x.shape
    return f(VP(x.data_ptr()), M, N, VP(offs.data_ptr()) if offs is not None else None,
             0 if offs is None else offs.numel(), *(VP(t.data_ptr()) for t in out),
             VP(stream.cuda_stream))


def _nan_columns(M, N, seed):
    """N(0,1) with colwise blocks that hold NaN: one whole 32x1 block of NaN
    (its 32x1 scale comes from no finite element) and single NaNs of either
    sign in otherwise finite blocks."""
    x = W.normal_bf16((M, N), seed=seed)
    x[32:64, 5] = 0x7FC0
    x[96 + 3, 7] = 0xFFC1
    x[M - 1, N - 2] = 0x7F81
    return x


def _cases():
    return [
        (W.moe_grouped(M=4096, N=2048, experts=8, routed_units=28, seed=3), "moe"),
        ((W.dual_specials(2048, 1024, seed=4), np.array([0, 1024, 1024, 1920], np.int32)),
         "specials"),
        ((_nan_columns(1024, 768, seed=5), None), "nan-columns dense"),
    ]


def test_noalloc_matches_oracle_and_workspace_form_on_calls_in_a_row():
    f = _noalloc_entry()
    stream = torch.cuda.current_stream()
    for (x_np, offs_np), tag in _cases():
        M, N = x_np.shape
        x = to_dev_bf16(x_np)
        offs = None if offs_np is None else torch.from_numpy(offs_np).cuda()
        got = _outputs(M, N)
        rc = _call(f, x, offs, got, stream)
        assert rc == mxq.OK, mxq.status_string(rc)
        ref = mxq.quantize_2d_dual_3pass(
            x, offs, workspace=torch.empty(M * N // 32, dtype=torch.uint8, device="cuda"),
            out=_outputs(M, N))
        torch.cuda.synchronize()
        g = _bytes(got)
        assert_dual_equal(g, oracle.mxfp8_dual_3pass(x_np, offs_np), f"{tag} vs oracle: ")
        assert_dual_equal(g, _bytes(ref), f"{tag} vs workspace form: ")


def test_noalloc_in_a_global_mode_graph_capture_replayed_on_fresh_inputs():
    f = _noalloc_entry()
    M, N = 2048, 1024
    offs_np = np.array([256, 256, 1536], np.int32)
    x = to_dev_bf16(W.normal_bf16((M, N), seed=11))
    offs = torch.from_numpy(offs_np).cuda()
    out = _outputs(M, N)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        # the first call on the device looks up the static array; it comes
        # before the capture, as the header asks
        assert _call(f, x, offs, out, side) == mxq.OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="global"):
        rc = _call(f, x, offs, out, side)
    assert rc == mxq.OK, mxq.status_string(rc)
    for seed in (12, 13):
        x_np = _nan_columns(M, N, seed) if seed == 13 else W.normal_bf16((M, N), seed=seed)
        x.copy_(to_dev_bf16(x_np))
        for t in out:
            t.fill_(FILL)
        g.replay()
        torch.cuda.synchronize()
        assert_dual_equal(_bytes(out), oracle.mxfp8_dual_3pass(x_np, offs_np),
                          f"replay with seed {seed}: ")


def test_noalloc_rejects_problems_beyond_its_scratch():
    f = _noalloc_entry()
    M, N = 32768, 16512            # M*N/32 is just above 16 MiB
    assert M * N // 32 > SCRATCH_BYTES
    fake = [VP(1 << 20)] * 4       # never dereferenced: rejected on the host
    assert f(VP(1 << 20), M, N, None, 0, *fake, None) == MXQ_ESCRATCH
    assert "scratch" in mxq.status_string(MXQ_ESCRATCH)
