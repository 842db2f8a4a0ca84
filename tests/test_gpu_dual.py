"""GPU parity of the dual-axis MXFP8 cast (mxq_quantize_2d_dual) against the CPU
oracle: every byte of q_row, s_row, q_col and s_col, on the published workloads
and on the edge cases the method has.  Destinations start filled with 0xAB so an
unwritten byte cannot pass."""
import math

import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq
import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.gpu_util import (FILL, assert_bytes_equal, assert_dual_equal, dual_outputs,
                            require_gpu, run_dual, to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _check(bits, offs, fill=FILL, tag=""):
    got = run_dual(bits, offs, fill)
    want = oracle.mxfp8_dual(bits, None if offs is None else np.asarray(offs, np.int32))
    assert_dual_equal(got, want, tag)
    return got


# --------------------------------------------------------------------------- workloads

def test_small_128x128_one_group():
    """128x128 bf16 N(0,1), offs = [128]."""
    x, offs = W.dual_small()
    _check(x, offs)


@pytest.mark.parametrize("M,N,offs", [
    (256, 384, None),
    (384, 256, [256, 256, 384]),               # an empty group
    (1024, 1024, [0, 128, 128, 512, 896]),    # empty groups + 128-row tail
    (1152, 2176, None),                        # 153 tiles: one more than the SM count
    (128, 20480, [128]),                       # 160 tiles in one tile row
    (2048, 128, [0, 0, 0, 2048]),              # leading empty groups
    (512, 512, [0]),                           # everything is uncovered tail
    (640, 384, [128, 640]),
])
def test_shapes_and_groups(M, N, offs):
    x = W.normal_bf16((M, N), seed=M * 7 + N)
    _check(x, offs, tag=f"{M}x{N} ")


def test_specials_8192x8192_dense():
    """Dense 8192x8192 with per-band scales 2^u, u in [-30, 15], zero/subnormal
    blocks and 0.01% +-Inf / 0.01% NaN: scale bytes 0, 254 and 255 all occur."""
    x = W.dual_specials()
    got = _check(x, None)
    for byte in (0, 254, 255):
        assert (got["s_col"] == byte).any() or (got["s_row"] == byte).any(), byte
    assert (got["s_col"] == 254).any() and (got["s_row"] == 255).any()


def test_moe_grouped_65536x7168():
    """MoE grouped: 64 groups of 128*Multinomial(448, 1/64) rows, offs[-1] = 57344,
    an 8192-row tail; destinations prefilled with 0xAB."""
    x, offs = W.moe_grouped()
    assert offs[-1] == 57344
    got = _check(x, offs)
    N = x.shape[1]
    assert not got["s_col"][N * 57344 // 32:].any()


@pytest.mark.parametrize("M,N", [(1024, 1024), (4096, 4096), (16384, 8192)])
def test_sweep_shapes_full(M, N):
    x = W.normal_bf16((M, N), seed=1)
    _check(x, None, tag=f"{M}x{N} ")


def test_sweep_largest_sampled():
    """32768x16384: every output byte of eight sampled 128-row tile rows, each
    checked against the oracle run on that slice alone (tiles are independent;
    for a dense group the slice's colwise atoms sit at stride M/128 atoms)."""
    M, N = 32768, 16384
    x = W.normal_bf16((M, N), seed=2)
    got = run_dual(x, None)
    TM = M // 128
    q_row = got["q_row"].reshape(M, N)
    q_col = got["q_col"].reshape(N, M)
    s_row = got["s_row"].reshape(TM, N // 128, 512)
    s_col = got["s_col"].reshape(N // 128, TM, 512)
    for ti in (0, 1, 77, 128, 200, 255, 256 - 3, TM - 1):
        sl = np.ascontiguousarray(x[128 * ti:128 * ti + 128])
        ref = oracle.mxfp8_dual(sl, None)
        assert_bytes_equal(q_row[128 * ti:128 * ti + 128], ref["q_row"], f"tile row {ti} q_row")
        assert_bytes_equal(s_row[ti], ref["s_row"], f"tile row {ti} s_row")
        assert_bytes_equal(q_col[:, 128 * ti:128 * ti + 128], ref["q_col"], f"tile row {ti} q_col")
        assert_bytes_equal(s_col[:, ti], ref["s_col"], f"tile row {ti} s_col")
    for k in got:
        assert not (got[k] == FILL).all()


# --------------------------------------------------------------------------- edge cases

def _golden_blocks():
    from tests.test_oracle_mxfp8_pins import _parse_overrides, _read_rows
    out = []
    for line in _read_rows("mxfp8_blocks.txt"):
        left = line.split("|")[0].split()
        blk = np.full(32, int(left[1], 16), np.uint16)
        for k, v in _parse_overrides(left[2]).items():
            blk[k] = v
        out.append(blk)
    return out


def test_edge_blocks_both_axes():
    """The page's special blocks (cutoff neighbours, scale byte 0 with the 2^127
    multiplier, Inf rowwise/colwise, NaN, -0, 2^127 next to -Inf) placed both as
    1x32 row blocks and as 32x1 column blocks of one tensor."""
    M = N = 256
    x = W.normal_bf16((M, N), seed=3)
    blocks = _golden_blocks()
    for t, blk in enumerate(blocks):
        r, c = divmod(t, N // 32)
        x[r, 32 * c:32 * c + 32] = blk                 # a row block in rows 0..
        x[128 + 32 * (t % 4):128 + 32 * (t % 4) + 32, 3 * t + 1] = blk  # a column block
    for t, amax in enumerate((0x0460, 0x0461, 0x045F, 0x04E0, 0x04E1, 0x0001, 0x007F, 0x0080)):
        blk = np.full(32, 0x0001, np.uint16)
        blk[5] = amax
        x[100, 32 * t:32 * t + 32] = blk
    _check(x, None)
    _check(x, [128, 128, 256])


def test_every_bf16_pattern():
    """All 65536 bf16 bit patterns (NaN payloads, +-Inf, subnormals, -0) shuffled
    into a 512x512 tensor, four times over with different shuffles."""
    g = np.random.Generator(np.random.PCG64(4))
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = np.concatenate([g.permutation(pats) for _ in range(4)]).reshape(512, 512)
    _check(x, None)
    _check(x, [256, 384])


def test_sparse_specials_keep_blocks_finite():
    """Mostly finite blocks with rare Inf/NaN and wide magnitudes: only the
    poisoned blocks change."""
    g = np.random.Generator(np.random.PCG64(5))
    xf = g.standard_normal((1024, 1024)).astype(np.float32) * np.exp2(
        g.integers(-130, 125, (1024, 1))).astype(np.float32)
    x = W.f32_to_bf16_bits(xf)
    flat = x.reshape(-1)
    idx = g.choice(flat.size, 200, replace=False)
    flat[idx[:100]] = 0x7F80 | (g.integers(0, 2, 100).astype(np.uint16) << 15)
    flat[idx[100:]] = 0x7FC1
    _check(x, [512, 1024])


def test_max_group_count():
    """G = 1024 groups (many empty) over 262144 rows, tail of 128 rows."""
    M, N = 262144, 128
    g = np.random.Generator(np.random.PCG64(6))
    units = np.sort(g.integers(0, M // 128, size=mxq.MAX_GROUPS))
    units[-1] = M // 128 - 1
    offs = (units * 128).astype(np.int32)
    x = W.normal_bf16((M, N), seed=6)
    _check(x, offs)


@pytest.mark.parametrize("offs", [
    [256, 128],          # not ascending
    [100, 256],          # not a multiple of 128
    [128, 384],          # beyond M
    [-128, 256],         # negative
])
def test_invalid_offsets_write_nothing(offs):
    M, N = 256, 256
    x = W.normal_bf16((M, N), seed=7)
    mxq.device_status(clear=True)
    got = run_dual(x, np.array(offs, np.int32))
    for k, v in got.items():
        assert (v == FILL).all(), f"{k} was written despite invalid offs"
    assert mxq.device_status(clear=True) & mxq.DEV_BADOFFS


def test_dirty_destinations_and_determinism():
    x, offs = W.moe_grouped(M=2048, N=1024, experts=8, routed_units=12)
    ref = oracle.mxfp8_dual(x, offs)
    for fill in (0x00, 0xFF, 0xAB, 0x7F):
        assert_dual_equal(run_dual(x, offs, fill), ref, f"fill {fill:#x} ")


def test_empty_problem_is_noop():
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    out = mxq.quantize_2d_dual(x)
    assert out.q_row.numel() == 0


def test_host_rejections_through_binding():
    base = torch.zeros(128 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    x = base[8:].view(128, 128)  # 16-byte offset: aligned
    mxq.quantize_2d_dual(x)
    x_bad = base[4:4 + 128 * 128].view(128, 128)  # 8-byte offset
    with pytest.raises(mxq.MxqError) as e:
        mxq.quantize_2d_dual(x_bad)
    assert e.value.code == mxq.EALIGN
    with pytest.raises(mxq.MxqError) as e:
        mxq.quantize_2d_dual(torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == mxq.EBADSHAPE
    with pytest.raises(mxq.MxqError) as e:
        mxq.quantize_2d_dual(torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda"),
                             torch.zeros(mxq.MAX_GROUPS + 1, dtype=torch.int32, device="cuda"))
    assert e.value.code == mxq.EBADOFFS


def test_side_stream_and_graph_capture():
    """The launch honours the caller's stream, so it captures into a CUDA graph;
    replaying the graph into 0xAB-filled buffers reproduces the outputs (an empty
    capture would leave the fill in place)."""
    x_np, offs_np = W.moe_grouped(M=1024, N=512, experts=4, routed_units=6)
    ref = oracle.mxfp8_dual(x_np, offs_np)
    x = to_dev_bf16(x_np)
    offs = torch.from_numpy(offs_np).cuda()
    out = dual_outputs(*x_np.shape)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mxq.quantize_2d_dual(x, offs, out=out, stream=s)  # warm-up on the side stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mxq.quantize_2d_dual(x, offs, out=out, stream=s)
    for t in out:
        t.fill_(FILL)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert_dual_equal({k: getattr(out, k).cpu().numpy().reshape(-1) for k in out._fields}, ref,
                      "graph ")


# --------------------------------------------------------------------------- layout pin

def _e4m3_table():
    return np.array([oracle.e4m3_value(c) if (c & 0x7F) != 0x7F else 0.0 for c in range(256)])


def _dequant(q: np.ndarray, scale_blocked: np.ndarray, R: int, K: int) -> np.ndarray:
    """Decode q [R, K] with its blocked [R, K/32] scales (reshape formulation)."""
    from tests.test_oracle_mxfp8_pins import _unblock_by_reshape
    s = _unblock_by_reshape(scale_blocked, R, K // 32).astype(np.int64)
    v = _e4m3_table()[q.reshape(R, K)]
    return v * np.exp2(np.repeat(s, 32, axis=1) - 127.0)


def _scaled_mm(a_u8, sa_u8, b_u8, sb_u8):
    """cuBLAS block-scaled MXFP8 GEMM: a [R, K] @ b [P, K]^T with blocked E8M0 scales."""
    e8 = getattr(torch, "float8_e8m0fnu", None)
    if e8 is None:
        pytest.skip("torch has no float8_e8m0fnu")
    a = a_u8.view(torch.float8_e4m3fn)
    b = b_u8.view(torch.float8_e4m3fn)
    try:
        return torch._scaled_mm(a, b.t(), sa_u8.view(e8), sb_u8.view(e8), out_dtype=torch.float32)
    except (RuntimeError, NotImplementedError) as err:
        pytest.skip(f"block-scaled _scaled_mm unavailable here: {err}")


def _close(got, a, b):
    """got ~ a @ b.T up to fp32 accumulation: |err| <= K * 2^-22 * (|a| @ |b|.T)."""
    ref = a @ b.T
    bound = np.abs(a) @ np.abs(b).T
    err = np.abs(got - ref)
    K = a.shape[1]
    assert np.all(err <= K * 2.0 ** -22 * bound + 1e-30), float((err / (bound + 1e-30)).max())
    assert np.abs(ref).max() > 0


def test_layout_pin_against_cublas_block_scaled_gemm():
    """Library-routine pin of the blocked scale layouts and the K-group slabs:
    cuBLAS's MXFP8 GEMM, fed the kernel's q/scale bytes, equals an fp64 GEMM of
    the same bytes decoded with the 128x4 layout.  Rowwise: x1 @ x2^T over N.
    Colwise: per K-group slab, x1[lo:hi]^T @ x2[lo:hi] over M."""
    M, N1, N2 = 1024, 256, 384
    offs = np.array([256, 256, 768], np.int32)   # groups [0,256), empty, [256,768), tail
    x1 = W.normal_bf16((M, N1), seed=11)
    x2 = W.normal_bf16((M, N2), seed=12)
    o1 = run_dual(x1, offs)
    o2 = run_dual(x2, offs)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()

    # rowwise: [M, N1] x [M, N1]^T (contraction over N1)
    got = _scaled_mm(dev(o1["q_row"].reshape(M, N1)), dev(o1["s_row"]),
                     dev(o1["q_row"].reshape(M, N1)), dev(o1["s_row"])).cpu().double().numpy()
    a = _dequant(o1["q_row"], o1["s_row"], M, N1)
    _close(got, a, a)

    # colwise, per group slab: [N1, G] x [N2, G]^T (contraction over the group's rows)
    lo = 0
    for hi in offs:
        if hi > lo:
            Gk = hi - lo
            qa = o1["q_col"].reshape(N1, M)[:, lo:hi]
            qb = o2["q_col"].reshape(N2, M)[:, lo:hi]
            sa = o1["s_col"][N1 * lo // 32:N1 * hi // 32]
            sb = o2["s_col"][N2 * lo // 32:N2 * hi // 32]
            got = _scaled_mm(dev(qa), dev(sa), dev(qb), dev(sb)).cpu().double().numpy()
            _close(got, _dequant(qa, sa, N1, Gk), _dequant(qb, sb, N2, Gk))
        lo = hi


def test_two_streams_at_once():
    """Two casts (and an MX9 pack) in flight on two streams at the same time each
    give the oracle's bytes: the calls share no scratch state."""
    xa, oa = W.moe_grouped(M=4096, N=1024, experts=8, routed_units=24, seed=41)
    xb = W.dual_specials(2048, 2048, seed=42)
    xm = W.mx9_outliers(1024, 1024, seed=43)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    da, db, dm = to_dev_bf16(xa), to_dev_bf16(xb), torch.from_numpy(xm).cuda()
    offs = torch.from_numpy(oa).cuda()
    torch.cuda.synchronize()
    outs_a, outs_b = dual_outputs(4096, 1024, FILL), dual_outputs(2048, 2048, FILL)
    with torch.cuda.stream(sa):
        mxq.quantize_2d_dual(da, offs, out=outs_a, stream=sa)
        q, e, p = mxq.mx9_pack(dm, stream=sa)
    with torch.cuda.stream(sb):
        mxq.quantize_2d_dual(db, None, out=outs_b, stream=sb)
    torch.cuda.synchronize()
    for got, x, o, tag in ((outs_a, xa, oa, "stream a "), (outs_b, xb, None, "stream b ")):
        want = oracle.mxfp8_dual(x, o)
        assert_dual_equal({k: getattr(got, k).cpu().numpy().reshape(-1) for k in got._fields}, want, tag)
    rq, re, rp = oracle.mx9_pack(xm)
    assert_bytes_equal(q.cpu().numpy().view(np.uint8), rq.view(np.uint8), "mx9 q on stream a")
    assert_bytes_equal(e.cpu().numpy(), re, "mx9 max_exp on stream a")


@pytest.mark.parametrize("i", range(32))
def test_random_shapes_and_groups(i):
    """32 seeded configurations: M and N multiples of 128 up to 2560 (tile counts
    on both sides of the SM count), dense or 1-12 groups with empty groups,
    leading empty groups and uncovered tails; values from per-band scales with
    zero, subnormal and non-finite blocks in some cases."""
    g = np.random.Generator(np.random.PCG64(2000 + i))
    M = 128 * int(g.integers(1, 21))
    N = 128 * int(g.integers(1, 21))
    if g.random() < 0.25:
        offs = None
    else:
        G = int(g.integers(1, 13))
        cuts = np.sort(g.integers(0, M // 128 + 1, size=G)) * 128
        if g.random() < 0.5:
            cuts[-1] = M  # no tail
        offs = [int(c) for c in cuts]
    x = W.normal_bf16((M, N), seed=3000 + i, scale=float(2.0 ** g.integers(-20, 20)))
    if i % 4 == 3:  # specials: a zero block row, subnormals, +-Inf and NaN
        x = x.copy()
        x[:32, :] = 0
        r = g.integers(0, M, size=8)
        c = g.integers(0, N, size=8)
        x[r[:2], c[:2]] = 0x7F80          # +Inf
        x[r[2:4], c[2:4]] = 0xFF80        # -Inf
        x[r[4:6], c[4:6]] = 0x7FC1        # NaN
        x[r[6:], c[6:]] = 0x0001          # smallest subnormal
    _check(x, offs, tag=f"case {i}: {M}x{N} offs {offs} ")
