"""GPU parity of the three-pass composition the fused cast replaces: the 1x32
cast, the 32x1 cast (NaN skipped by its amax), the K-groups scale swizzle and
the composed call, each byte-exact against the CPU oracle; plus the one
documented divergence from the fused cast (NaN in a colwise block)."""
import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import FILL, assert_bytes_equal, assert_dual_equal, require_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _filled(shape):
    return torch.full(shape, FILL, dtype=torch.uint8, device="cuda")


def _run_3pass(x_np, offs_np):
    M, N = x_np.shape
    x = to_dev_bf16(x_np)
    o = None if offs_np is None else torch.from_numpy(np.asarray(offs_np, np.int32)).cuda()
    out = mxq.DualOutputs(_filled((M, N)), _filled((M * N // 32,)), _filled((N, M)),
                          _filled((M * N // 32,)))
    ws = _filled((M * N // 32,))
    mxq.quantize_2d_dual_3pass(x, o, workspace=ws, out=out)
    torch.cuda.synchronize()
    got = {k: getattr(out, k).cpu().numpy().reshape(-1) for k in out._fields}
    got["s_rm"] = ws.cpu().numpy()
    return got


def _check_3pass(x_np, offs_np, tag=""):
    got = _run_3pass(x_np, offs_np)
    want = oracle.mxfp8_dual_3pass(x_np, None if offs_np is None else np.asarray(offs_np, np.int32))
    assert_dual_equal(got, want, tag)
    assert_bytes_equal(got["s_rm"], want["s_rm"], tag + "s_rm")
    return got


@pytest.mark.parametrize("M,N,offs", [
    (128, 128, [128]),
    (256, 384, None),
    (1024, 1024, [0, 128, 128, 512, 896]),
    (1152, 2176, None),
    (512, 512, [0]),
])
def test_three_pass_shapes(M, N, offs):
    _check_3pass(W.normal_bf16((M, N), seed=M + 3 * N), offs, f"{M}x{N} ")


def test_three_pass_every_bf16_pattern():
    """All bf16 patterns: the 32x1 cast's NaN-skipping amax and saturating Inf."""
    g = np.random.Generator(np.random.PCG64(8))
    x = np.concatenate([g.permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16))
                        for _ in range(4)]).reshape(512, 512)
    _check_3pass(x, [256, 384])


def test_three_pass_moe_65536x7168():
    x, offs = W.moe_grouped()
    _check_3pass(x, offs)


def test_single_axis_entry_points():
    M, N = 640, 384
    x_np = W.dual_specials(M, N, seed=9)
    x = to_dev_bf16(x_np)
    q_row, s_row = mxq.quantize_1x32(x)
    q_col, s_rm = mxq.quantize_32x1(x)
    torch.cuda.synchronize()
    r = oracle.mxfp8_1x32(x_np)
    c = oracle.mxfp8_32x1(x_np)
    assert_bytes_equal(q_row.cpu().numpy(), r["q_row"], "q_row")
    assert_bytes_equal(s_row.cpu().numpy(), r["s_row"], "s_row")
    assert_bytes_equal(q_col.cpu().numpy(), c["q_col"], "q_col")
    assert_bytes_equal(s_rm.cpu().numpy(), c["s_rm"], "s_rm")


def test_swizzle_alone_and_invalid_offsets():
    N, M = 384, 1024
    g = np.random.Generator(np.random.PCG64(10))
    s_rm = g.integers(0, 256, size=(N, M // 32), dtype=np.uint8)
    for offs in ([1024], [0, 256, 256, 768], None):
        o = None if offs is None else torch.tensor(offs, dtype=torch.int32, device="cuda")
        out = mxq.swizzle_kgroups(torch.from_numpy(s_rm).cuda(), o, out=_filled((N * M // 32,)))
        torch.cuda.synchronize()
        assert_bytes_equal(out.cpu().numpy(),
                           oracle.swizzle_kgroups(s_rm, None if offs is None else np.array(offs, np.int32)),
                           f"swizzle {offs}")
    mxq.device_status(clear=True)
    bad = torch.tensor([512, 256], dtype=torch.int32, device="cuda")
    out = mxq.swizzle_kgroups(torch.from_numpy(s_rm).cuda(), bad, out=_filled((N * M // 32,)))
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == FILL).all()
    assert mxq.device_status(clear=True) & mxq.DEV_BADOFFS


def test_fused_and_three_pass_differ_only_in_nan_columns():
    """The page's fused cast poisons a colwise block holding NaN (scale 255, all
    0x7F) where the 32x1 cast it replaces keeps the other elements' scale; the
    difference is asserted so that a change on either side fails loudly."""
    M, N = 256, 256
    x_np = W.normal_bf16((M, N), seed=13)
    x_np[37, 129] = 0x7FC0
    offs = [256]
    fused = oracle.mxfp8_dual(x_np, np.array(offs, np.int32))
    three = _check_3pass(x_np, offs)
    from tests.gpu_util import run_dual
    fused_gpu = run_dual(x_np, np.array(offs, np.int32))
    assert_dual_equal(fused_gpu, fused, "fused ")
    for k in ("q_row", "s_row"):
        assert np.array_equal(fused_gpu[k], three[k])
    qf = fused_gpu["q_col"].reshape(N, M)
    qt = three["q_col"].reshape(N, M)
    diff = np.argwhere(qf != qt)
    assert diff.size and set(diff[:, 0].tolist()) == {129} and diff[:, 1].max() < 64
    assert (qf[129, 32:64] == 0x7F).all() and (qt[129, 32:64] == 0x7F).sum() == 1
    assert (fused_gpu["s_col"] != three["s_col"]).sum() == 1


def test_three_pass_rejections():
    x = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mxq.MxqError) as e:
        mxq.quantize_2d_dual_3pass(x, workspace=torch.zeros(100, dtype=torch.uint8, device="cuda"))
    assert e.value.code == mxq.EBADSHAPE
    with pytest.raises(mxq.MxqError) as e:
        mxq.quantize_1x32(torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == mxq.EBADSHAPE
