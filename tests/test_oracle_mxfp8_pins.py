"""Pins of the CPU oracle's MXFP8 half against facts that do not come from the oracle.

Each test names the mistake it is there to catch.  Sources:
* pytorch/ao PR #4995 "Fused dual-axis MXFP8 quantization with correct metadata"
  (description, review replies) -- printed cutoff, non-finite rules, the
  uncovered tail, per-group unblocking as the check of the scale placement.
* the OCP FP8 E4M3 format, through PyTorch's float8_e4m3fn cast (a library
  routine: round-to-nearest-even for |v| <= 448).
* the 128x4 blocked scale layout, restated as a tensor reshape/permute.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.conftest import golden_path


def _read_rows(name):
    rows = []
    with open(golden_path(name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def _bf16_val(bits: int) -> float:
    return float(W.bf16_bits_to_f32(np.array([bits], np.uint16))[0])


# ---------------------------------------------------------------------------
# E8M0 rceil scale
# ---------------------------------------------------------------------------

def test_scale_cutoff_printed_value():
    """The page's cutoff 448*2^-127 is fp32 0x04600000; neighbours land on bytes 0/1.

    Catches: a wrong constant (448 vs 480/256), a wrong bias, '<' for '<='.
    """
    cutoff = np.array([448.0 * 2.0 ** -127], np.float32)
    assert cutoff.view(np.uint32)[0] == 0x04600000
    for line in _read_rows("mxfp8_scale_cutoff.txt"):
        bits, want = line.split()
        assert oracle.e8m0_rceil(_bf16_val(int(bits, 16))) == int(want), line


def test_scale_powers_of_two_closed_form():
    """amax = 2^k -> s = k + 119 (1.75*2^(s-127-... )); amax = 448*2^j -> s = j + 127.

    Catches: off-by-one in the exponent, rounding the scale down instead of up.
    """
    for k in range(-119, 128):
        assert oracle.e8m0_rceil(math.ldexp(1.0, k)) == k + 119, k
    for k in range(-140, -119):
        assert oracle.e8m0_rceil(math.ldexp(1.0, k)) == 0, k
    for j in range(-127, 121):
        v = math.ldexp(448.0, j)
        assert oracle.e8m0_rceil(v) == j + 127, j
        up = math.ldexp(448.0 + 2.0, j)  # next bf16 value above 448*2^j
        assert oracle.e8m0_rceil(up) == j + 128, j


def test_scale_exhaustive_against_bit_formula():
    """All 32640 finite non-negative bf16 amax values: the definition equals an
    independently derived integer formula on the bf16 bits,
    s = max(0, E - 8 + [mantissa > 0x60]) with E the exponent field.

    Catches: any disagreement between the definition and its bit-level form,
    including subnormal amax and the largest finite value (s = 247).
    """
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # all finite non-negative bf16
    E = (bits >> 7).astype(np.int64)
    f = (bits & 0x7F).astype(np.int64)
    want = np.maximum(0, E - 8 + (f > 0x60))
    vals = W.bf16_bits_to_f32(bits.astype(np.uint16)).astype(np.float64)
    got = np.array([oracle.e8m0_rceil(v) for v in vals])
    np.testing.assert_array_equal(got, want)
    assert got.max() == 247


def test_scale_is_minimal_and_sufficient():
    """For every finite bf16 amax: amax/2^(s-127) <= 448 and, for s > 0,
    amax/2^(s-128) > 448 (the scale cannot be lowered without saturating)."""
    bits = np.arange(0, 0x7F80, 7, dtype=np.uint16)
    for v in W.bf16_bits_to_f32(bits).astype(np.float64):
        s = oracle.e8m0_rceil(v)
        assert v <= math.ldexp(448.0, s - 127)
        if s > 0:
            assert v > math.ldexp(448.0, s - 128)


# ---------------------------------------------------------------------------
# E4M3 encoding
# ---------------------------------------------------------------------------

def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_code_table_matches_torch():
    """Decoding every finite code agrees with PyTorch's float8_e4m3fn -> float32,
    and encode(decode(c)) == c.  Catches: wrong bias, wrong subnormal step."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    mine = np.array([oracle.e4m3_value(int(c)) for c in codes])
    np.testing.assert_array_equal(mine, ref.astype(np.float64))
    for c in codes:
        assert oracle.e4m3_encode(oracle.e4m3_value(int(c))) == c
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_all_bf16_in_range_matches_torch():
    """Every bf16 value with |v| <= 448 encodes as PyTorch's RNE cast does.

    Catches: truncation instead of rounding, a wrong rounding boundary, a lost sign.
    """
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    v = W.bf16_bits_to_f32(bits)
    keep = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[keep]
    np.testing.assert_array_equal(oracle.e4m3_encode_array(v), _torch_e4m3(v))


def test_e4m3_encode_ties_to_even_matches_torch():
    """Exact midpoints between neighbouring codes, and their fp32 neighbours.

    Catches: ties away from zero, ties to odd.
    """
    vals = sorted({oracle.e4m3_value(c) for c in range(0x7F)})
    pts = []
    for a, b in zip(vals[:-1], vals[1:]):
        mid = np.float32((a + b) / 2.0)
        assert float(mid) == (a + b) / 2.0
        pts += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
    pts = np.array(pts + [-p for p in pts], np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode_array(pts), _torch_e4m3(pts))


def test_e4m3_saturation_and_specials():
    """Closed forms of the saturating cast: +-Inf and finite overflow -> +-448, NaN -> 0x7F."""
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-449.0) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-(2.0 ** -11)) == 0x80  # rounds to -0
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00     # tie with 0 -> even (0)
    assert oracle.e4m3_encode(3 * 2.0 ** -11) == 0x01


# ---------------------------------------------------------------------------
# one block: the page's non-finite and scale-0 rules
# ---------------------------------------------------------------------------

def _parse_overrides(s):
    out = {}
    if s != "-":
        for kv in s.split(","):
            k, v = kv.split("=")
            out[int(k)] = int(v, 16)
    return out


@pytest.mark.parametrize("line", _read_rows("mxfp8_blocks.txt"))
def test_block_golden(line):
    """Hand-derived blocks for the rules the page states (fixture cites them)."""
    left, scale, data = [t.strip() for t in line.split("|")]
    axis, fill, over = left.split()
    x = np.full(32, int(fill, 16), np.uint16)
    for k, v in _parse_overrides(over).items():
        x[k] = v
    dfill, dover = data.split()
    want = np.full(32, int(dfill, 16), np.uint8)
    for k, v in _parse_overrides(dover).items():
        want[k] = v
    if axis == "col32x1":
        s, q = oracle.mxfp8_block_nan_dropped(x)
    else:
        s, q = oracle.mxfp8_block(x, colwise=(axis == "col"))
    assert s == int(scale)
    np.testing.assert_array_equal(q, want)


def test_block_dequant_error_bound():
    """For random finite blocks over a wide exponent range the data byte is the
    nearest point of the scaled E4M3 grid: |q*2^(s-127) - x| is at most half
    the local grid step, and nothing saturates.

    Catches: a scale one too large (precision loss beyond the bound) or too
    small (saturation), wrong multiplier sign, a dropped 2^127 at byte 0.
    """
    g = np.random.Generator(np.random.PCG64(7))
    for trial in range(400):
        e = int(g.integers(-140, 120))
        x = (g.standard_normal(32) * 2.0 ** e).astype(np.float32)
        bits = W.f32_to_bf16_bits(x)
        xv = W.bf16_bits_to_f32(bits).astype(np.float64)
        for colwise in (False, True):
            s, q = oracle.mxfp8_block(bits, colwise)
            assert s < 254
            for xi, qi in zip(xv, q):
                y = math.ldexp(oracle.e4m3_value(int(qi)), s - 127)
                a = abs(xi) * 2.0 ** (127 - s)
                assert a <= 448.0
                # grid step at |v|: 2^-9 below 2^-6, else 2^(floor(log2 a) - 3)
                step = 2.0 ** -9 if a < 2.0 ** -6 else 2.0 ** (math.floor(math.log2(a)) - 3)
                assert abs(y - xi) <= math.ldexp(step / 2, s - 127), (xi, y, s)
                if xi != 0:
                    assert math.copysign(1, y) == math.copysign(1, xi) or y == 0


def test_block_value_idempotent():
    """dequant(quant(dequant(quant x))) == dequant(quant x): the grid is closed."""
    g = np.random.Generator(np.random.PCG64(3))
    for _ in range(300):
        x = W.f32_to_bf16_bits(g.standard_normal(32).astype(np.float32) * np.float32(2.0 ** int(g.integers(-60, 60))))
        s, q = oracle.mxfp8_block(x, False)
        y = np.array([math.ldexp(oracle.e4m3_value(int(c)), s - 127) for c in q], np.float32)
        yb = W.f32_to_bf16_bits(y)
        assert np.array_equal(W.bf16_bits_to_f32(yb), y)  # dequantized values fit bf16
        s2, q2 = oracle.mxfp8_block(yb, False)
        y2 = np.array([math.ldexp(oracle.e4m3_value(int(c)), s2 - 127) for c in q2])
        np.testing.assert_array_equal(y2, y.astype(np.float64))


# ---------------------------------------------------------------------------
# layouts and whole-tensor assembly
# ---------------------------------------------------------------------------

def _blocked_by_reshape(mat: torch.Tensor) -> torch.Tensor:
    """The 128x4 blocked layout as a reshape: atoms row-block-major, inside an
    atom [32 (r % 32)] x [4 (r // 32 % 4)] x [4 (c % 4)]."""
    R, C = mat.shape
    t = mat.reshape(R // 128, 128, C // 4, 4).permute(0, 2, 1, 3)
    t = t.reshape(-1, 4, 32, 4).transpose(1, 2)
    return t.reshape(-1)


def _unblock_by_reshape(flat: np.ndarray, R: int, C: int) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(flat)).reshape(R // 128, C // 4, 32, 4, 4)
    return t.permute(0, 3, 2, 1, 4).reshape(R, C).numpy()


@pytest.mark.parametrize("R,C", [(128, 4), (256, 8), (384, 12), (128, 32), (512, 4)])
def test_blocked_index_matches_reshape_formulation(R, C):
    """Every (r, c) lands where the reshape formulation puts it; atoms are 512 B."""
    ids = torch.arange(R * C, dtype=torch.int64).reshape(R, C)
    flat = _blocked_by_reshape(ids).numpy()
    for r in range(R):
        for c in range(C):
            assert flat[oracle.blocked_index(r, c, R, C)] == r * C + c
    assert oracle.blocked_index(127, 3, R, C) == 511
    assert oracle.blocked_index(0, 4, R, C) == (512 if C > 4 else 512 * 1)
    np.testing.assert_array_equal(_unblock_by_reshape(flat, R, C), ids.numpy())


def _check_dual_against_blocks(x, offs, out):
    """Rebuild every output from the oracle's single-block function plus the
    reshape-based unblocking (the page's 'per-group unblocking' check)."""
    M, N = x.shape
    q_row = out["q_row"].reshape(M, N)
    q_col = out["q_col"].reshape(N, M)
    s_row = _unblock_by_reshape(out["s_row"], M, N // 32)
    for m in range(M):
        for j in range(N // 32):
            s, q = oracle.mxfp8_block(x[m, 32 * j:32 * j + 32], False)
            assert s_row[m, j] == s
            np.testing.assert_array_equal(q_row[m, 32 * j:32 * j + 32], q)
    col_s = np.zeros((N, M // 32), np.uint8)
    for i in range(M // 32):
        for n in range(N):
            s, q = oracle.mxfp8_block(np.ascontiguousarray(x[32 * i:32 * i + 32, n]), True)
            col_s[n, i] = s
            np.testing.assert_array_equal(q_col[n, 32 * i:32 * i + 32], q)
    ends = [M] if offs is None else list(offs)
    lo = 0
    for hi in ends:
        if hi > lo:
            slab = out["s_col"][N * lo // 32:N * hi // 32]
            np.testing.assert_array_equal(
                _unblock_by_reshape(slab, N, (hi - lo) // 32), col_s[:, lo // 32:hi // 32])
        lo = hi
    assert not out["s_col"][N * ends[-1] // 32:].any()


@pytest.mark.parametrize("M,N,offs", [
    (128, 128, [128]),
    (128, 128, None),
    (256, 128, [128]),                      # uncovered tail of one tile row
    (512, 256, [0, 128, 128, 384]),         # empty groups and a tail
    (384, 256, [256, 256, 384]),
])
def test_dual_assembly(M, N, offs):
    x = W.normal_bf16((M, N), seed=M + N)
    o = None if offs is None else np.array(offs, np.int32)
    out = oracle.mxfp8_dual(x, o)
    _check_dual_against_blocks(x, offs, out)


def test_dense_equals_single_group():
    """offs = None is the one-group case offs = [M] (the page's dense placement)."""
    x = W.normal_bf16((256, 384), seed=5)
    a = oracle.mxfp8_dual(x, None)
    b = oracle.mxfp8_dual(x, np.array([256], np.int32))
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_tail_rows_quantized_and_scales_zero():
    """Rows past offs[-1] are still quantized in q_row, s_row and q_col; only their
    column scales are zero (page: 'Uncovered tail')."""
    x = W.normal_bf16((384, 128), seed=11)
    full = oracle.mxfp8_dual(x, None)
    part = oracle.mxfp8_dual(x, np.array([128], np.int32))
    for k in ("q_row", "s_row", "q_col"):
        np.testing.assert_array_equal(full[k], part[k])
    assert not part["s_col"][128 * 128 // 32:].any()
    assert part["s_col"][:128 * 128 // 32].all()


def test_block_independence():
    """Changing one 32x32 block changes only the outputs of the blocks it touches."""
    M, N = 256, 256
    x = W.normal_bf16((M, N), seed=2)
    a = oracle.mxfp8_dual(x, None)
    y = x.copy()
    y[64:96, 160:192] = W.normal_bf16((32, 32), seed=99, scale=1000.0)
    b = oracle.mxfp8_dual(y, None)
    qa, qb = a["q_row"].reshape(M, N), b["q_row"].reshape(M, N)
    mask = np.zeros((M, N), bool)
    mask[64:96, 160:192] = True
    assert np.array_equal(qa[~mask], qb[~mask])
    ca, cb = a["q_col"].reshape(N, M), b["q_col"].reshape(N, M)
    assert np.array_equal(ca[~mask.T], cb[~mask.T])
    sa = _unblock_by_reshape(a["s_row"], M, N // 32)
    sb = _unblock_by_reshape(b["s_row"], M, N // 32)
    smask = np.zeros_like(sa, bool)
    smask[64:96, 5] = True
    assert np.array_equal(sa[~smask], sb[~smask]) and not np.array_equal(sa[smask], sb[smask])


def test_zero_tensor():
    out = oracle.mxfp8_dual(np.zeros((128, 128), np.uint16), None)
    for k in out:
        assert not out[k].any()


@pytest.mark.parametrize("offs,M,ok", [
    (None, 256, True), ([256], 256, True), ([0, 0, 256], 256, True), ([128], 256, True),
    ([], 256, False), ([64], 256, False), ([256, 128], 256, False), ([384], 256, False),
    ([-128, 128], 256, False),
])
def test_offs_validation(offs, M, ok):
    o = None if offs is None else np.array(offs, np.int32)
    rc = oracle.check_offs(o, M) if offs != [] else oracle.check_offs(np.zeros(0, np.int32), M)
    assert (rc == oracle.OK) == ok


def test_bad_shapes_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.mxfp8_dual(np.zeros((100, 128), np.uint16), None)
    with pytest.raises(oracle.OracleError):
        oracle.mxfp8_dual(np.zeros((128, 96), np.uint16), None)


def test_bytes_per_element_closed_form():
    """Page: the fused kernel moves 4.0625 B per input element (2 in + 1 + 1 +
    1/32 + 1/32 out); the three-kernel composition moved 6.125."""
    M, N = 256, 384
    out = oracle.mxfp8_dual(np.zeros((M, N), np.uint16), None)
    moved = 2 * M * N + sum(v.size for v in out.values())
    assert moved / (M * N) == 4.0625
    # three kernels: two reads of x, the four outputs, and a read+write of the
    # colwise scales by the separate swizzle pass
    assert (2 * 2 * M * N + sum(v.size for v in out.values()) + 2 * (M * N // 32)) / (M * N) == 6.125


# ---------------------------------------------------------------------------
# the three-pass composition the fused cast replaces
# ---------------------------------------------------------------------------

def test_nan_dropped_rule_equals_colwise_rule_without_nan():
    """With no NaN in the block the separate 32x1 cast and the fused colwise
    rule agree (the page: the only divergence is NaN on the colwise output)."""
    g = np.random.Generator(np.random.PCG64(12))
    for _ in range(300):
        x = W.f32_to_bf16_bits((g.standard_normal(32) * 2.0 ** int(g.integers(-130, 120)))
                               .astype(np.float32))
        if g.random() < 0.3:
            x[int(g.integers(32))] = 0x7F80 | (int(g.integers(2)) << 15)
        a = oracle.mxfp8_block(x, True)
        b = oracle.mxfp8_block_nan_dropped(x)
        assert a[0] == b[0]
        np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("M,N,offs", [(256, 384, None), (512, 256, [0, 128, 128, 384]),
                                      (384, 128, [384]), (256, 256, [0])])
def test_swizzle_matches_reshape_blocking(M, N, offs):
    """The swizzle's slabs equal the reshape statement of the blocked layout
    applied to each group's columns; the tail is zero."""
    g = np.random.Generator(np.random.PCG64(M + N))
    s_rm = g.integers(0, 256, size=(N, M // 32), dtype=np.uint8)
    o = None if offs is None else np.array(offs, np.int32)
    out = oracle.swizzle_kgroups(s_rm, o)
    ends = [M] if offs is None else offs
    lo = 0
    for hi in ends:
        if hi > lo:
            want = _blocked_by_reshape(torch.from_numpy(np.ascontiguousarray(s_rm[:, lo // 32:hi // 32]))).numpy()
            np.testing.assert_array_equal(out[N * lo // 32:N * hi // 32], want)
        lo = hi
    assert not out[N * ends[-1] // 32:].any()


def test_three_pass_equals_fused_except_nan_columns():
    """The composition matches the fused cast byte for byte except in colwise
    blocks holding NaN, where the fused cast poisons (255, all 0x7F) and the
    composition keeps the other elements' scale."""
    M, N = 256, 256
    x = W.normal_bf16((M, N), seed=21)
    x[5, 7] = 0x7FC0          # NaN: row block (5, 0), column block (0, 7)
    x[100, 200] = 0x7F80      # +Inf: both rules agree
    offs = np.array([128, 256], np.int32)
    a = oracle.mxfp8_dual(x, offs)
    b = oracle.mxfp8_dual_3pass(x, offs)
    for k in ("q_row", "s_row"):
        np.testing.assert_array_equal(a[k], b[k])
    qa, qb = a["q_col"].reshape(N, M), b["q_col"].reshape(N, M)
    diff = np.argwhere(qa != qb)
    assert diff.size and set(map(tuple, diff[:, :1].tolist())) == {(7,)}
    assert np.all((diff[:, 1] >= 0) & (diff[:, 1] < 32))
    assert (qa[7, :32] == 0x7F).all() and qb[7, 5] == 0x7F and (qb[7, :32] != 0x7F).sum() == 31
    sa = _unblock_by_reshape(a["s_col"][:N * 128 // 32], N, 4)
    sb = _unblock_by_reshape(b["s_col"][:N * 128 // 32], N, 4)
    assert sa[7, 0] == 255 and sb[7, 0] < 255
    sa[7, 0] = sb[7, 0]
    np.testing.assert_array_equal(sa, sb)
    np.testing.assert_array_equal(a["s_col"][N * 128 // 32:], b["s_col"][N * 128 // 32:])
