"""Consumer check of the cast's layouts by a block-scaled MMA of this library:
mxq_mxfp8_scaled_mm (tcgen05.mma, kind mxf8f6f4, E8M0 scales per 32 K
elements) reads q_row/s_row, and a K-group's columns of q_col with that
group's s_col slab, in place (no copy or re-layout), and must equal an fp64
product of the same bytes decoded through the 128x4 blocked layout, up to
fp32 accumulation.  pytorch/ao PR #4995 (description, first paragraph, and the
"Uncovered tail" paragraph): the scales are written in the blocked form that
the block-scaled MMA consumes, the colwise ones one slab per K-group."""
import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import require_gpu, run_dual
from tests.test_gpu_dual import _close, _dequant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_one_tile_rowwise():
    """One 128x128 output tile, K = 128: q_row/s_row of one tensor against
    itself (the smallest product: one scale atom per operand)."""
    x = W.normal_bf16((128, 128), seed=21)
    o = run_dual(x, None)
    q = _dev(o["q_row"].reshape(128, 128))
    s = _dev(o["s_row"])
    got = mxq.mxfp8_scaled_mm(q, s, q, s).cpu().double().numpy()
    a = _dequant(o["q_row"], o["s_row"], 128, 128)
    _close(got, a, a)


def test_rowwise_and_grouped_colwise_in_place():
    """Rowwise over N: x1 @ x2^T with both tensors' q_row/s_row (several tiles
    and K steps).  Colwise per K-group: q_col[:, lo:hi] read in place with the
    group's s_col slab, against the same for a second tensor; an empty group
    and an uncovered tail are present."""
    M, N1, N2 = 1024, 384, 256
    offs = np.array([256, 256, 768], np.int32)
    x1 = W.normal_bf16((M, N1), seed=22)
    x2 = W.normal_bf16((M, N2), seed=23)
    o1, o2 = run_dual(x1, offs), run_dual(x2, offs)
    y1 = W.normal_bf16((512, N1), seed=24)
    oy = run_dual(y1, None)
    got = mxq.mxfp8_scaled_mm(_dev(o1["q_row"].reshape(M, N1)), _dev(o1["s_row"]),
                              _dev(oy["q_row"].reshape(512, N1)), _dev(oy["s_row"]))
    _close(got.cpu().double().numpy(), _dequant(o1["q_row"], o1["s_row"], M, N1),
           _dequant(oy["q_row"], oy["s_row"], 512, N1))

    qc1 = _dev(o1["q_col"].reshape(N1, M))
    qc2 = _dev(o2["q_col"].reshape(N2, M))
    sc1, sc2 = _dev(o1["s_col"]), _dev(o2["s_col"])
    lo = 0
    for hi in offs:
        if hi > lo:
            g = hi - lo
            got = mxq.mxfp8_scaled_mm(qc1[:, lo:hi], sc1[N1 * lo // 32:N1 * hi // 32],
                                      qc2[:, lo:hi], sc2[N2 * lo // 32:N2 * hi // 32])
            qa = o1["q_col"].reshape(N1, M)[:, lo:hi]
            qb = o2["q_col"].reshape(N2, M)[:, lo:hi]
            _close(got.cpu().double().numpy(),
                   _dequant(qa, o1["s_col"][N1 * lo // 32:N1 * hi // 32], N1, g),
                   _dequant(qb, o2["s_col"][N2 * lo // 32:N2 * hi // 32], N2, g))
        lo = hi


def test_scales_across_the_exponent_range():
    """Rows scaled by 2^u, u from -30 to 15 per 32-row band (the specials
    workload's scaling without its non-finite values): scale bytes far from
    127 on both operands must reach the MMA unchanged."""
    x = W.dual_specials(512, 256, seed=25)
    bits = x.copy()
    bad = (bits & 0x7F80) == 0x7F80          # drop Inf/NaN: the product is then finite
    bits[bad] = 0
    o = run_dual(bits, None)
    q, s = _dev(o["q_row"].reshape(512, 256)), _dev(o["s_row"])
    got = mxq.mxfp8_scaled_mm(q, s, q, s).cpu().double().numpy()
    a = _dequant(o["q_row"], o["s_row"], 512, 256)
    _close(got, a, a)


def test_rejections():
    q = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros(128 * 128 // 32, dtype=torch.uint8, device="cuda")
    with pytest.raises(mxq.MxqError):
        mxq.mxfp8_scaled_mm(q[:, :96], s[:384], q[:, :96], s[:384])   # K not a multiple of 128
    with pytest.raises(ValueError):
        mxq.mxfp8_scaled_mm(q, s, q[:, :64], s)                         # K mismatch
