"""Tensors past 2^31 elements (the largest sizes the calls take without any
32-bit index): the dual-axis cast, dense and grouped with a tail, and MX9
pack/unpack.  Inputs are drawn on the device (seeded); sampled tile rows (and
rows) are checked byte for byte against the oracle run on those slices alone,
which tiles and blocks being independent makes exact."""
import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from tests.gpu_util import FILL, assert_bytes_equal, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    torch.cuda.empty_cache()
    assert mxq.device_status(clear=True) == 0


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("grouped", [False, True])
def test_dual_past_2_31_elements(grouped):
    M, N = 32768, 65664  # M*N = 2,151,677,952 > 2^31
    assert M * N > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(21)
    x = (torch.randn(M, N, device="cuda", generator=g, dtype=torch.bfloat16) * 0.02)
    offs_np = np.array([M // 2, M - 256], np.int32) if grouped else None
    offs = None if offs_np is None else torch.from_numpy(offs_np).cuda()
    kw = dict(dtype=torch.uint8, device="cuda")
    out = mxq.DualOutputs(torch.full((M, N), FILL, **kw), torch.full((M * N // 32,), FILL, **kw),
                          torch.full((N, M), FILL, **kw), torch.full((M * N // 32,), FILL, **kw))
    mxq.quantize_2d_dual(x, offs, out=out)
    torch.cuda.synchronize()
    TM, TN = M // 128, N // 128
    s_row = out.s_row.view(TM, TN, 512)
    for ti in (0, 1, TM // 2 - 1, TM // 2, TM - 3, TM - 1):
        r0 = 128 * ti
        sl = _bits(x[r0:r0 + 128])
        ref = oracle.mxfp8_dual(sl, None)
        tag = f"tile row {ti} "
        assert_bytes_equal(out.q_row[r0:r0 + 128].cpu().numpy(), ref["q_row"], tag + "q_row")
        assert_bytes_equal(s_row[ti].cpu().numpy(), ref["s_row"], tag + "s_row")
        assert_bytes_equal(out.q_col[:, r0:r0 + 128].cpu().numpy(), ref["q_col"], tag + "q_col")
        # the slice's colwise atom tj is the tile's atom in the full s_col
        lo, hi, end = 0, M, M
        if grouped:
            end = int(offs_np[-1])
            lo = 0 if r0 < offs_np[0] else int(offs_np[0])
            hi = int(offs_np[0]) if r0 < offs_np[0] else int(offs_np[1])
        atoms = ref["s_col"].reshape(TN, 512)
        s_col = out.s_col.cpu().numpy()
        for tj in (0, 1, TN // 2, TN - 1):
            if r0 < end:
                at = N * lo // 32 + (tj * ((hi - lo) // 128) + (r0 - lo) // 128) * 512
                assert_bytes_equal(s_col[at:at + 512], atoms[tj], tag + f"s_col atom {tj}")
            else:
                at = N * end // 32 + (((r0 - end) // 128) * TN + tj) * 512
                assert (s_col[at:at + 512] == 0).all(), tag + f"tail atom {tj}"
    # every scale byte is written (0xAB is no scale these data can produce)
    assert bool((out.s_row != FILL).all()) and bool((out.s_col != FILL).all())


def test_mx9_past_2_31_elements():
    rows, cols = 131072, 16400  # 2,149,580,800 elements
    assert rows * cols > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(22)
    x = torch.randn(rows, cols, device="cuda", generator=g)
    q, e, p = mxq.mx9_pack(x)
    y = mxq.mx9_unpack(q, e, p, torch.float32, (rows, cols))
    torch.cuda.synchronize()
    bpr = cols // 16
    for r in (0, 1, rows // 2, rows - 2, rows - 1):
        xr = x[r:r + 1].cpu().numpy()
        rq, re, rp = oracle.mx9_pack(xr)
        assert_bytes_equal(q[r * bpr:(r + 1) * bpr].cpu().numpy().view(np.uint8), rq.view(np.uint8),
                           f"row {r} q")
        assert_bytes_equal(e[r * bpr:(r + 1) * bpr].cpu().numpy(), re, f"row {r} max_exp")
        assert_bytes_equal(p[r * bpr:(r + 1) * bpr].cpu().numpy().reshape(-1), rp.reshape(-1),
                           f"row {r} prime")
        ry = oracle.mx9_unpack(rq, re, rp, "f32", 1, cols)
        assert_bytes_equal(y[r].cpu().view(torch.int32).numpy().view(np.uint8),
                           ry.view(np.uint8), f"row {r} unpack")


@pytest.mark.parametrize("axis", [1, 0])
def test_packed_mx9_past_2_31_elements(axis):
    rows, cols = 131072, 16400
    g = torch.Generator(device="cuda").manual_seed(23)
    x = torch.randn(rows, cols, device="cuda", generator=g)
    rec = mxq.mx_pack_packed(x, mxq.FMT_MX9, axis)
    y = torch.empty_like(x)
    mxq.mx_unpack_packed(rec, mxq.FMT_MX9, y, axis)
    torch.cuda.synchronize()
    if axis == 1:
        bpl = cols // 16
        for r in (0, rows // 2, rows - 1):
            want = oracle.mx_pack(x[r:r + 1].cpu().numpy(), mxq.FMT_MX9, axis=1)
            assert_bytes_equal(rec[r * bpl:(r + 1) * bpl].cpu().numpy(), want, f"row {r} records")
            ry = oracle.mx_unpack(want, mxq.FMT_MX9, 1, cols, "f32", axis=1)
            assert_bytes_equal(y[r].cpu().view(torch.int32).numpy().view(np.uint8),
                               ry.view(np.uint8), f"row {r} unpack")
    else:
        bpl = rows // 16
        for c in (0, cols // 2, cols - 1):
            xc = np.ascontiguousarray(x[:, c:c + 1].cpu().numpy())
            want = oracle.mx_pack(xc, mxq.FMT_MX9, axis=0)
            assert_bytes_equal(rec[c * bpl:(c + 1) * bpl].cpu().numpy(), want, f"column {c} records")
            ry = oracle.mx_unpack(want, mxq.FMT_MX9, rows, 1, "f32", axis=0)
            got = np.ascontiguousarray(y[:, c:c + 1].cpu().numpy())
            assert_bytes_equal(got.view(np.uint8), ry.view(np.uint8), f"column {c} unpack")
