"""Bands of rows (data-parallel shards along M) of the dual-axis cast: every
band's outputs are the full tensor's bytes at the band's places, and bands that
cover [0, M) once fill the full colwise scale buffer exactly once, with no
exchange between them.  Compared with the CPU oracle of the full tensor."""
import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import FILL, assert_bytes_equal, require_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _bands_check(x_np, offs_np, cuts, order=None):
    M, N = x_np.shape
    want = oracle.mxfp8_dual(x_np, offs_np)
    offs = None if offs_np is None else torch.from_numpy(offs_np).cuda()
    s_col = torch.full((N * M // 32,), FILL, dtype=torch.uint8, device="cuda")
    xd = to_dev_bf16(x_np)
    edges = [0] + list(cuts) + [M]
    bands = list(zip(edges[:-1], edges[1:]))
    got = {}
    for lo, hi in (bands if order is None else [bands[i] for i in order]):
        kw = dict(dtype=torch.uint8, device="cuda")
        out = (torch.full((hi - lo, N), FILL, **kw), torch.full(((hi - lo) * N // 32,), FILL, **kw),
               torch.full((N, hi - lo), FILL, **kw))
        got[lo] = mxq.quantize_2d_dual_rows(xd[lo:hi], lo, M, s_col, offs, out=out)
    torch.cuda.synchronize()
    q_row = want["q_row"].reshape(M, N)
    q_col = want["q_col"].reshape(N, M)
    for lo, hi in bands:
        o = got[lo]
        tag = f"band [{lo}, {hi}) "
        assert_bytes_equal(o.q_row.cpu().numpy().reshape(-1), q_row[lo:hi].reshape(-1), tag + "q_row")
        assert_bytes_equal(o.s_row.cpu().numpy(), want["s_row"][lo * N // 32:hi * N // 32], tag + "s_row")
        assert_bytes_equal(o.q_col.cpu().numpy().reshape(-1),
                           np.ascontiguousarray(q_col[:, lo:hi]).reshape(-1), tag + "q_col")
    assert_bytes_equal(s_col.cpu().numpy(), want["s_col"], "s_col (all bands)")


def test_bands_of_the_grouped_workload():
    """Groups split by band edges, groups ending on them, empty groups and the
    uncovered tail across two bands."""
    x, _ = W.moe_grouped(M=2048, N=512, experts=8, routed_units=14, seed=5)
    offs = np.array([256, 256, 640, 896, 1024, 1408, 1536, 1792], np.int32)
    _bands_check(x, offs, cuts=[512, 1152, 1664])


def test_bands_in_any_order_and_dense():
    x = W.dual_specials(1024, 384, seed=6)
    _bands_check(x, None, cuts=[128, 640], order=[2, 0, 1])
    _bands_check(x, np.array([384, 1024], np.int32), cuts=[256, 768], order=[1, 2, 0])


def test_one_band_is_the_full_call():
    x, offs = W.moe_grouped(M=1024, N=256, experts=4, routed_units=6, seed=7)
    _bands_check(x, offs, cuts=[])
