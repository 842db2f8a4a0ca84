"""GPU parity of MX9/MX6 in one packed tensor (mx_pack_packed / mx_unpack_packed)
against the CPU oracle, byte for byte: both formats, fp32 and bf16, blocks
along either axis, strided (wider) rows, zero-padded partial blocks."""
import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import assert_bytes_equal, require_gpu

pytestmark = pytest.mark.gpu

FMTS = [mxq.FMT_MX9, mxq.FMT_MX6]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(x_full: np.ndarray, cols: int, fmt: int, axis: int, tag: str):
    """x_full: [rows, ld] host array whose first `cols` columns are the tensor."""
    rows, ld = x_full.shape
    xd = _dev(x_full)[:, :cols]                      # a strided view when ld > cols
    got = mxq.mx_pack_packed(xd, fmt, axis)
    want = oracle.mx_pack(x_full, fmt, axis=axis, cols=cols)
    torch.cuda.synchronize()
    assert_bytes_equal(got.cpu().numpy(), want, f"{tag} pack")
    # unpack into a prefilled wider buffer: only the tensor's elements change
    is_bf16 = x_full.dtype == np.uint16
    fill_val = 0x5A5A if is_bf16 else np.float32(-3.25)
    fill = np.full((rows, ld), fill_val, x_full.dtype)
    yd = _dev(fill)
    mxq.mx_unpack_packed(got, fmt, yd[:, :cols], axis)
    ref = oracle.mx_unpack(want, fmt, rows, cols, "bf16" if is_bf16 else "f32", axis=axis, ld=ld,
                           fill=fill)
    torch.cuda.synchronize()
    ygot = yd.cpu().view(torch.int16 if is_bf16 else torch.int32).numpy()
    assert_bytes_equal(ygot.view(np.uint8), ref.view(np.uint8), f"{tag} unpack")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("rows,cols,ld", [(64, 256, 256), (20, 37, 37), (48, 80, 112),
                                          (33, 16, 24), (1, 15, 15), (257, 129, 136),
                                          (3, 16, 16), (7, 48, 48), (1000, 160, 160),
                                          (1, 4096, 4096), (129, 2048, 2048),
                                          (40, 512, 528), (33, 2048, 2064), (5, 4096, 4224)])
def test_packed_shapes(fmt, dt, axis, rows, cols, ld):
    x = np.zeros((rows, ld), np.float32)
    x[:, :cols] = W.mx9_outliers(rows, cols, seed=rows * cols + axis, zero_blocks=0, tiny_blocks=0)
    x[:, cols:] = np.float32(9e30)                   # outside the tensor: must not matter
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    _check(x, cols, fmt, axis, f"fmt{fmt} {dt} axis{axis} {rows}x{cols}/{ld}")


def _tma_cols_geometry(fmt: int, dt: str, rows: int, ld: int) -> bool:
    """Blocks along columns move as TMA tiles when the row pitch and each
    column's records are multiples of 16 bytes (pointers here are aligned)."""
    rec = 18 if fmt == mxq.FMT_MX9 else 12
    return (ld * (2 if dt == "bf16" else 4)) % 16 == 0 and (-(-rows // 16) * rec) % 16 == 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols,ld", [(120, 37, 40), (120, 38, 40), (248, 36, 40),
                                          (128, 300, 304), (113, 8, 8), (1020, 700, 704),
                                          (2048, 1000, 1000), (4096, 4096, 4096), (60, 1, 8),
                                          (250, 129, 136), (3968, 2304, 2312)])
def test_packed_cols_tma_tiles(fmt, dt, rows, cols, ld):
    """Blocks along columns through the TMA tiles: ragged columns and rows
    (partial tiles and blocks), padded pitches, several tiles per CTA."""
    if not _tma_cols_geometry(fmt, dt, rows, ld):
        pytest.skip("geometry outside the TMA tiles for this format")
    x = np.zeros((rows, ld), np.float32)
    x[:, :cols] = W.mx9_outliers(rows, cols, seed=rows + 7 * cols, zero_blocks=0, tiny_blocks=0)
    x[:, cols:] = np.float32(-7e33)                  # outside the tensor: must not matter
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    _check(x, cols, fmt, 0, f"fmt{fmt} {dt} axis0 {rows}x{cols}/{ld}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(1, 16), (129, 16), (1, 32), (257, 32), (128, 16)])
def test_packed_last_group_of_few_records(fmt, dt, rows, cols):
    """Contiguous whole-block rows through the record kernels where the last
    group of 128 records holds one or two records (MX6: 12 or 24 bytes, less
    than or not a multiple of a 16-byte unit), or the whole tensor is one record."""
    x = W.mx9_outliers(rows, cols, seed=rows + cols, zero_blocks=0, tiny_blocks=0)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    _check(x, cols, fmt, 1, f"fmt{fmt} {dt} {rows}x{cols}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("axis", [0, 1])
def test_packed_outlier_workload(fmt, axis):
    """The [4096, 4096] outlier workload (zero and ~1e-40 blocks included)."""
    x = W.mx9_outliers()
    _check(x, 4096, fmt, axis, f"fmt{fmt} axis{axis} 4096^2")


@pytest.mark.parametrize("fmt", FMTS)
def test_packed_every_bf16_pattern(fmt):
    g = np.random.Generator(np.random.PCG64(3))
    x = g.permutation(np.arange(65536, dtype=np.uint32).astype(np.uint16)).reshape(256, 256)
    _check(x, 256, fmt, 1, f"fmt{fmt} bf16 patterns")
    _check(x, 256, fmt, 0, f"fmt{fmt} bf16 patterns axis0")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("rows,cols", [(512, 1024), (129, 200)])
def test_packed_tiny_exponent_blocks(fmt, dt, axis, rows, cols):
    """Blocks of subnormals and the smallest normals, where the scale exponent is
    clamped at -126 and a subnormal element can round to a nonzero code."""
    x = W.tiny_exponents(rows, cols, dt == "bf16", seed=rows + 7 * axis + fmt)
    _check(x, cols, fmt, axis, f"fmt{fmt} {dt} axis{axis} tiny {rows}x{cols}")


def test_packed_mx9_matches_split_kernel():
    """The packed MX9 records hold the split kernels' bytes (GPU against GPU)."""
    x = _dev(W.mx9_outliers(512, 512, seed=5))
    rec = mxq.mx_pack_packed(x, mxq.FMT_MX9, 1)
    q, e, p = mxq.mx9_pack(x)
    torch.cuda.synchronize()
    r = rec.cpu().numpy()
    assert np.array_equal(r[:, 0], e.cpu().numpy())
    assert np.array_equal(r[:, 1], p.cpu().numpy()[:, 0])
    assert np.array_equal(r[:, 2:].view(np.int8), q.cpu().numpy())


def test_packed_rejections():
    with pytest.raises(ValueError):
        mxq.mx_pack_packed(torch.zeros((4, 16), device="cuda"), 7, 1)       # unknown format
    with pytest.raises(ValueError):
        mxq.mx_pack_packed(torch.zeros((4, 16), device="cuda").t(), mxq.FMT_MX9, 1)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("x_off,p_off", [(1, 0), (0, 1)])
def test_packed_offsets_below_16_bytes(fmt, dt, x_off, p_off):
    """Element pointers one element off 16 bytes, or records at the smallest
    allowed offset (2 bytes for MX9, 4 for MX6): the contiguous row-blocked
    case then runs without its 16-byte vector paths and gives the same bytes."""
    rows, cols = 64, 512
    x = W.mx9_outliers(rows, cols, seed=21, zero_blocks=0, tiny_blocks=0)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    rb, nb = mxq.RECORD_BYTES[fmt], rows * cols // 16
    want = oracle.mx_pack(x, fmt, axis=1)
    flat = np.concatenate([np.zeros(x_off, x.dtype), x.reshape(-1)])  # data from element x_off
    xd = _dev(flat)[x_off:x_off + rows * cols].view(rows, cols)
    poff = (2 if fmt == mxq.FMT_MX9 else 4) * p_off
    big = torch.zeros(nb * rb + 16, dtype=torch.uint8, device="cuda")
    pk = big[poff:poff + nb * rb]
    mxq.mx_pack_packed(xd, fmt, 1, out=pk)
    torch.cuda.synchronize()
    assert_bytes_equal(pk.cpu().numpy().reshape(nb, rb), want, f"fmt{fmt} {dt} pack offsets")
    is_bf16 = dt == "bf16"
    fill = np.full(rows * cols + 1, 0x5A5A if is_bf16 else np.float32(-3.25), x.dtype)
    yd_big = _dev(fill)
    yd = yd_big[x_off:x_off + rows * cols].view(rows, cols)
    mxq.mx_unpack_packed(pk, fmt, yd, 1)
    ref = oracle.mx_unpack(want, fmt, rows, cols, "bf16" if is_bf16 else "f32", axis=1)
    torch.cuda.synchronize()
    got = yd.cpu().view(torch.int16 if is_bf16 else torch.int32).numpy()
    assert_bytes_equal(got.view(np.uint8), ref.view(np.uint8), f"fmt{fmt} {dt} unpack offsets")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("axis,pitch", [(1, 0), (1, 64), (0, 0), (0, 8)])
def test_packed_calls_replay_in_a_cuda_graph(fmt, axis, pitch):
    """After one eager call (which sets up each kernel), pack and unpack record
    into a CUDA graph and its replay gives the eager bytes."""
    rows, cols = 256, 1024
    wide = _dev(W.normal_f32((rows, cols + pitch), seed=31))
    x = wide[:, :cols]
    rec = mxq.mx_pack_packed(x, fmt, axis)
    y = torch.empty_like(wide)[:, :cols]
    mxq.mx_unpack_packed(rec, fmt, y, axis)
    torch.cuda.synchronize()
    rec_eager, y_eager = rec.clone(), y.clone()
    rec.zero_()
    y.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mxq.mx_pack_packed(x, fmt, axis, out=rec, stream=s)
        mxq.mx_unpack_packed(rec, fmt, y, axis, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(rec, rec_eager)
    assert torch.equal(y.contiguous().view(torch.int32), y_eager.contiguous().view(torch.int32))


def _fuzz_case(i: int):
    """Seeded geometry i.  Odd-numbered quarters of the cases are aligned (16-byte
    element and record offsets and pitches, whole 16-element blocks or sizes
    just under a tile) so that the vector, record and TMA kernels are reached;
    the others take arbitrary sizes, pitches and offsets."""
    g = np.random.Generator(np.random.PCG64(1000 + i))
    dt = ("f32", "bf16")[i % 2]
    fmt = FMTS[(i // 2) % 2]
    axis = (i // 4) % 2
    es = 4 if dt == "f32" else 2
    if (i // 8) % 2:  # aligned
        unit = 16 // es  # elements per 16 bytes
        run = 128 if fmt == mxq.FMT_MX9 else 64  # rows whose records fill 16-byte runs
        rows = int(run * g.integers(1, 5) - g.integers(0, 16))
        cols = int(16 * g.integers(1, 40)) if g.random() < 0.5 else int(unit * g.integers(1, 90))
        pad = int(unit * g.choice([0, 0, 1, 2, 5]))
        x_off = int(unit * g.choice([0, 1]))
        p_off = int(g.choice([0, 8]))  # 0 or 16 / 32 bytes
    else:
        rows = int(g.integers(1, 400))
        cols = int(g.integers(1, 700))
        pad = int(g.choice([0, 0, 1, 3, 4, 8, 16, 37]))
        x_off = int(g.choice([0, 0, 1, 4, 8]))
        p_off = int(g.choice([0, 0, 1, 8]))  # in units of the record alignment (2 or 4 bytes)
    return dt, fmt, axis, rows, cols, pad, x_off, p_off


@pytest.mark.parametrize("i", range(64))
def test_packed_random_geometries(i):
    """64 seeded geometries through whichever kernel each one selects (TMA
    column tiles, vector or element column tiles, record rows, generic rows):
    records and the unpacked tensor equal the oracle, and nothing outside the
    tensor's elements (pitch padding, the bytes before an offset view) changes."""
    dt, fmt, axis, rows, cols, pad, x_off, p_off = _fuzz_case(i)
    is_bf16 = dt == "bf16"
    pitch = cols + pad
    xs = W.mx9_outliers(rows, cols, seed=i, zero_blocks=0, tiny_blocks=0)
    full = np.full((rows, pitch), np.float32(-6e35), np.float32)
    full[:, :cols] = xs
    if is_bf16:
        full = W.f32_to_bf16_bits(full)
    want = oracle.mx_pack(full, fmt, axis=axis, cols=cols)
    flat = np.concatenate([np.zeros(x_off, full.dtype), full.reshape(-1)])
    xd = _dev(flat)[x_off:].view(rows, pitch)[:, :cols]
    rb = mxq.RECORD_BYTES[fmt]
    nb = want.shape[0]
    poff = (2 if fmt == mxq.FMT_MX9 else 4) * p_off
    big = torch.full((nb * rb + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    pk = big[poff:poff + nb * rb]
    tag = f"case {i}: {dt} fmt{fmt} axis{axis} {rows}x{cols} pitch {pitch} x_off {x_off} p_off {poff}"
    mxq.mx_pack_packed(xd, fmt, axis, out=pk)
    torch.cuda.synchronize()
    bcpu = big.cpu().numpy()
    assert_bytes_equal(bcpu[poff:poff + nb * rb].reshape(nb, rb), want, tag + " pack")
    assert (bcpu[:poff] == 0xAB).all() and (bcpu[poff + nb * rb:] == 0xAB).all(), tag + " outside records"
    fill = np.full(x_off + rows * pitch, 0x5A5A if is_bf16 else np.float32(-3.25), full.dtype)
    yflat = _dev(fill)
    yd = yflat[x_off:].view(rows, pitch)[:, :cols]
    mxq.mx_unpack_packed(pk, fmt, yd, axis)
    ref = oracle.mx_unpack(want, fmt, rows, cols, "bf16" if is_bf16 else "f32", axis=axis,
                           ld=pitch, fill=fill[x_off:].reshape(rows, pitch))
    torch.cuda.synchronize()
    got = yflat.cpu().view(torch.int16 if is_bf16 else torch.int32).numpy()
    assert_bytes_equal(got[x_off:].view(np.uint8), ref.view(np.uint8), tag + " unpack")
    assert np.array_equal(got[:x_off], fill[:x_off].view(got.dtype)), tag + " before the view"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("rem", [1, 2, 3, 31, 33, 127])
@pytest.mark.parametrize("pad", [0, 64])
def test_packed_record_group_remainders(fmt, dt, rem, pad):
    """Rows of an odd number c of whole blocks, with rows chosen so that the
    block count leaves `rem` records in the last 128-record group (and so a
    partial last run of the record pack's 32- and 128-block runs); pad 64: the
    same with strided rows (c >= 129 blocks, the strided record kernels)."""
    g = np.random.Generator(np.random.PCG64(97 * rem + 7 * pad + fmt + (dt == "bf16")))
    c = int(g.integers(129, 320)) | 1 if pad else int(g.integers(1, 64)) * 2 + 1
    rows = (rem * pow(c, -1, 128)) % 128 + 128 * int(g.integers(0, 3))
    rows = rows or 128
    assert (rows * c) % 128 == rem % 128
    cols = 16 * c
    x = np.zeros((rows, cols + pad), np.float32)
    x[:, :cols] = W.mx9_outliers(rows, cols, seed=rem + rows, zero_blocks=0, tiny_blocks=0)
    x[:, cols:] = np.float32(3e33)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    _check(x, cols, fmt, 1, f"fmt{fmt} {dt} {rows}x{cols}/{cols + pad} rem {rem}")
