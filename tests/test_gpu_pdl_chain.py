"""Ordering across programmatic dependent launch.

Every kernel of the library is launched so that it may be scheduled while its
stream predecessor still runs, and waits for that predecessor before its first
global access.  These tests chain kernels whose inputs are the previous
kernel's outputs, in one stream and in a captured CUDA graph (where the edges
between the kernels are programmatic), and check the final bytes against the
oracle: a kernel that read its input early would see stale or partial data.

The MX9 round trip is idempotent after its first pass (pack(unpack(pack x)) =
pack x, pinned on the oracle), so a chain of pack/unpack pairs must end where
one pair ends; the dual cast then reads the last unpack's bf16 output directly.
"""
import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import FILL, assert_bytes_equal, assert_dual_equal, dual_outputs, require_gpu

pytestmark = pytest.mark.gpu

ROWS, COLS = 1024, 2048
ROUNDS = 12


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _expected():
    """Oracle: one bf16 MX9 round trip of the input, then the dual cast of it."""
    xb = W.f32_to_bf16_bits(W.mx9_outliers(ROWS, COLS, seed=31, zero_blocks=8, tiny_blocks=8))
    q, e, p = oracle.mx9_pack(xb)
    yb = oracle.mx9_unpack(q, e, p, "bf16", ROWS, COLS)
    # the round trip is a fixed point from here on
    q2, e2, p2 = oracle.mx9_pack(yb)
    assert np.array_equal(q2, q) and np.array_equal(e2, e) and np.array_equal(p2, p)
    return xb, yb, (q, e, p), oracle.mxfp8_dual(yb.view(np.uint16), None)


def _chain(x, y, q, e, p, out, stream):
    """ROUNDS pack/unpack pairs feeding each other, then the dual cast of y."""
    src = x
    for _ in range(ROUNDS):
        mxq.mx9_pack(src, out=(q, e, p), stream=stream)
        mxq.mx9_unpack(q, e, p, torch.bfloat16, (ROWS, COLS), out=y, stream=stream)
        src = y
    mxq.quantize_2d_dual(y, out=out, stream=stream)


def _buffers(xb):
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    nb = ROWS * COLS // 16
    q = torch.full((nb, 16), -1, dtype=torch.int8, device="cuda")
    e = torch.full((nb,), FILL, dtype=torch.uint8, device="cuda")
    p = torch.full((nb, 1), FILL, dtype=torch.uint8, device="cuda")
    y = torch.full((ROWS, COLS), float("nan"), dtype=torch.bfloat16, device="cuda")
    return x, y, q, e, p, dual_outputs(ROWS, COLS)


def _check(y, q, e, p, out, yb, qep, dual):
    assert_bytes_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), yb.view(np.uint16), "y")
    for got, want, name in zip((q, e, p), qep, ("q", "max_exp", "prime")):
        assert_bytes_equal(got.cpu().numpy(), want, name)
    assert_dual_equal({k: getattr(out, k).cpu().numpy().reshape(-1) for k in out._fields}, dual,
                      "dual of the chained output: ")


def test_chain_on_one_stream():
    xb, yb, qep, dual = _expected()
    x, y, q, e, p, out = _buffers(xb)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _chain(x, y, q, e, p, out, s)
    torch.cuda.synchronize()
    _check(y, q, e, p, out, yb, qep, dual)


def test_chain_in_a_graph_replayed_after_new_input():
    xb, yb, qep, dual = _expected()
    x, y, q, e, p, out = _buffers(xb)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _chain(x, y, q, e, p, out, s)  # first calls outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _chain(x, y, q, e, p, out, s)
    # poison every intermediate and output, then replay: every byte must be rebuilt
    for t, v in ((y, float("nan")), (q, -1), (e, FILL), (p, FILL)):
        t.fill_(v)
    for t in out:
        t.fill_(FILL)
    g.replay()
    torch.cuda.synchronize()
    _check(y, q, e, p, out, yb, qep, dual)
