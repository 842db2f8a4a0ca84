"""GPU parity of MX9 pack/unpack (mx9_pack, mx9_unpack) against the CPU oracle:
q, max_exp, prime and the rebuilt tensor, bit for bit, for fp32 and bf16."""
import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import assert_bytes_equal, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _dev(x: np.ndarray) -> torch.Tensor:
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _fill_like(shape, dtype, byte=0xAB):
    t = torch.empty(shape, dtype=dtype, device="cuda")
    t.view(torch.uint8).fill_(byte)
    return t


def _check_pack_unpack(x: np.ndarray, tag=""):
    rows, cols = x.shape
    nb = rows * cols // 16
    out = (_fill_like((nb, 16), torch.int8), _fill_like((nb,), torch.uint8),
           _fill_like((nb, 1), torch.uint8))
    q, e, p = mxq.mx9_pack(_dev(x), out=out)
    rq, re, rp = oracle.mx9_pack(x)
    torch.cuda.synchronize()
    assert_bytes_equal(q.cpu().numpy().view(np.uint8), rq.view(np.uint8), f"{tag}q")
    assert_bytes_equal(e.cpu().numpy(), re, f"{tag}max_exp")
    assert_bytes_equal(p.cpu().numpy(), rp, f"{tag}prime")
    for out_dtype, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
        y = _fill_like((rows, cols), out_dtype)
        mxq.mx9_unpack(q, e, p, out_dtype, (rows, cols), out=y)
        ry = oracle.mx9_unpack(rq, re, rp, name, rows, cols)
        torch.cuda.synchronize()
        got = y.cpu().view(torch.int32 if name == "f32" else torch.int16).numpy()
        assert_bytes_equal(got.view(np.uint8), ry.view(np.uint8), f"{tag}unpack {name}")


def test_outliers_4096x4096_fp32():
    """[4096, 4096] N(0,1), 1% x100, 64 zero and 64 ~1e-40 blocks, fp32."""
    _check_pack_unpack(W.mx9_outliers(), "fp32 ")


def test_outliers_4096x4096_bf16():
    """The same tensor rounded to bf16."""
    _check_pack_unpack(W.mx9_outliers_bf16(), "bf16 ")


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 16), (1, 32), (7, 48), (1000, 160),
                                        (33, 4096), (4097, 64)])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_ragged_shapes(rows, cols, dt):
    x = W.mx9_outliers(rows, cols, seed=rows + cols, zero_blocks=0, tiny_blocks=0)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    _check_pack_unpack(x, f"{rows}x{cols} {dt} ")


def test_every_bf16_pattern():
    g = np.random.Generator(np.random.PCG64(1))
    x = np.concatenate([g.permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16))
                        for _ in range(2)]).reshape(512, 256)
    _check_pack_unpack(x, "bf16 patterns ")


def test_random_fp32_bit_patterns_and_ties():
    """Random fp32 bit patterns (NaN, Inf, subnormals included), plus exact
    rounding ties and the +-128 boundary of demoted pairs."""
    g = np.random.Generator(np.random.PCG64(2))
    x = g.integers(0, 2 ** 32, size=(512, 512), dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = x.copy()
    ties = np.float32(1.0) + np.arange(1, 129, dtype=np.float32) * np.float32(2.0 ** -7)
    x[0, :128] = ties                                   # x / 2^k lands on .5 steps
    x[1, :16] = np.float32(1.0)
    x[1, 2:4] = np.float32(0.99999)                     # demoted pair near 128 steps
    x[2, :16] = np.float32(0.75 * 2.0 ** -126)          # subnormals that round to 1
    _check_pack_unpack(x, "fp32 bits ")


@pytest.mark.parametrize("M,N", [(1024, 1024), (4096, 4096), (16384, 8192)])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_sweep_shapes_full(M, N, dt):
    x = W.normal_f32((M, N), seed=3)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    _check_pack_unpack(x, f"{M}x{N} {dt} ")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_sweep_largest_sampled(dt):
    """32768x16384: blocks are independent along rows, so the oracle checks
    every output of 64 sampled rows; the rebuilt tensor is checked on them too."""
    M, N = 32768, 16384
    x = W.normal_f32((M, N), seed=4)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    q, e, p = mxq.mx9_pack(_dev(x))
    y = mxq.mx9_unpack(q, e, p, torch.float32 if dt == "f32" else torch.bfloat16, (M, N))
    torch.cuda.synchronize()
    rows = np.random.Generator(np.random.PCG64(5)).choice(M, 64, replace=False)
    rows[0], rows[1] = 0, M - 1
    bpr = N // 16
    for r in rows:
        rq, re, rp = oracle.mx9_pack(np.ascontiguousarray(x[r:r + 1]))
        assert_bytes_equal(q[r * bpr:(r + 1) * bpr].cpu().numpy().view(np.uint8),
                           rq.view(np.uint8), f"row {r} q")
        assert_bytes_equal(e[r * bpr:(r + 1) * bpr].cpu().numpy(), re, f"row {r} max_exp")
        assert_bytes_equal(p[r * bpr:(r + 1) * bpr].cpu().numpy(), rp, f"row {r} prime")
        ry = oracle.mx9_unpack(rq, re, rp, dt, 1, N)
        got = y[r].cpu().view(torch.int32 if dt == "f32" else torch.int16).numpy()
        assert_bytes_equal(got.view(np.uint8), ry.view(np.uint8), f"row {r} unpack")


def test_snr_of_device_roundtrip():
    """The device round trip reaches the page's quality (~46 dB clean)."""
    x = W.normal_f32((2048, 2048), seed=6)
    xt = _dev(x)
    q, e, p = mxq.mx9_pack(xt)
    y = mxq.mx9_unpack(q, e, p, torch.float32, x.shape)
    err = (y.double() - xt.double()).pow(2).sum()
    snr = 10 * torch.log10(xt.double().pow(2).sum() / err).item()
    assert abs(snr - 46.0) < 1.0


def test_rejections_through_binding():
    with pytest.raises(mxq.MxqError) as e:
        mxq.mx9_pack(torch.zeros((4, 15), device="cuda"))
    assert e.value.code == mxq.EBADSHAPE
    with pytest.raises(ValueError):
        mxq.mx9_pack(torch.zeros((4, 16), dtype=torch.float16, device="cuda"))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(256, 1024), (300, 1040)])
def test_unpack_with_unaligned_exponent_and_prime_pointers(rows, cols, dt):
    """max_exp and prime may start at any byte (the ABI asks alignment of q and
    the output only): byte-offset views give the oracle's bytes."""
    x = W.mx9_outliers(rows, cols, seed=11)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    nb = rows * cols // 16
    q, e, p = mxq.mx9_pack(_dev(x))
    e_big = torch.zeros(nb + 3, dtype=torch.uint8, device="cuda")
    p_big = torch.zeros(nb + 5, dtype=torch.uint8, device="cuda")
    e_big[3:].copy_(e)
    p_big[5:].copy_(p.reshape(-1))
    rq, re, rp = oracle.mx9_pack(x)
    for out_dtype, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
        y = _fill_like((rows, cols), out_dtype)
        mxq.mx9_unpack(q, e_big[3:], p_big[5:], out_dtype, (rows, cols), out=y)
        ry = oracle.mx9_unpack(rq, re, rp, name, rows, cols)
        torch.cuda.synchronize()
        got = y.cpu().view(torch.int32 if name == "f32" else torch.int16).numpy()
        assert_bytes_equal(got.view(np.uint8), ry.view(np.uint8), f"unaligned unpack {name}")


@pytest.mark.parametrize("i", range(16))
def test_random_shapes(i):
    """16 seeded shapes (1-600 rows, 16-2400 columns in whole blocks), fp32 and
    bf16, outlier data with zero and ~1e-40 blocks, through the split pack and
    unpack."""
    g = np.random.Generator(np.random.PCG64(4000 + i))
    rows = int(g.integers(1, 601))
    cols = 16 * int(g.integers(1, 151))
    nz = min(16, rows * cols // 16 // 8)  # zero and ~1e-40 blocks, as many as fit
    x = W.mx9_outliers(rows, cols, seed=5000 + i, zero_blocks=nz, tiny_blocks=nz)
    if i % 2:
        x = W.f32_to_bf16_bits(x)
    _check_pack_unpack(x, tag=f"case {i}: {rows}x{cols} {'bf16' if i % 2 else 'f32'} ")


@pytest.mark.parametrize("rows,cols", [(1, 16), (1, 32), (1, 48), (3, 48), (5, 80), (999, 48),
                                       (1000, 48), (4099, 4112)])
def test_unpack_output_tails(rows, cols):
    """The unpack stores whole 128-byte rows of output by tensor store and the
    bytes past the last whole row by lane stores (under 128 bytes: all of
    them).  These shapes leave 0, 32, 64 or 96 bytes past the last whole row
    for fp32 and bf16 output, from a 64-byte tensor up to one whose rounds
    wrap the grid several times; every byte is the oracle's."""
    nz = min(16, rows * cols // 16 // 8)
    x = W.mx9_outliers(rows, cols, seed=rows + cols, zero_blocks=nz, tiny_blocks=nz)
    _check_pack_unpack(x, tag=f"{rows}x{cols} ")


@pytest.mark.parametrize("offset_bytes", [16, 48, 112])
def test_unpack_into_an_output_at_a_16_byte_offset(offset_bytes):
    """The output may start at any 16-byte boundary (the tensor store's map is
    encoded on the pointer as given): an output view 16, 48 or 112 bytes into
    a larger buffer gets the oracle's bytes and nothing outside the view is
    written."""
    rows, cols = 129, 4096
    x = W.mx9_outliers(rows, cols, seed=offset_bytes, zero_blocks=8, tiny_blocks=8)
    q, e, p = mxq.mx9_pack(_dev(x))
    rq, re, rp = oracle.mx9_pack(x)
    for out_dtype, name, esize in ((torch.float32, "f32", 4), (torch.bfloat16, "bf16", 2)):
        n = rows * cols
        pad = offset_bytes // esize
        big = _fill_like((n + pad + 64,), out_dtype)
        y = big[pad:pad + n].view(rows, cols)
        mxq.mx9_unpack(q, e, p, out_dtype, (rows, cols), out=y)
        ry = oracle.mx9_unpack(rq, re, rp, name, rows, cols)
        torch.cuda.synchronize()
        raw = big.cpu().view(torch.uint8).numpy()
        lo, hi = offset_bytes, offset_bytes + n * esize
        assert_bytes_equal(raw[lo:hi], ry.view(np.uint8).reshape(-1), f"offset {offset_bytes} {name}")
        assert (raw[:lo] == 0xAB).all() and (raw[hi:] == 0xAB).all(), "bytes outside the view"
