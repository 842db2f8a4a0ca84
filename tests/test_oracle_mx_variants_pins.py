"""Pins of the oracle's MX9/MX6 single-packed-tensor path (any axis, strided,
zero-padded partial blocks) against facts that do not come from that path.

Source: AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
pack/unpack" (commits "pack mx9 into a single uint8 tensor and dispatch
mx6/mx9 to the packed kernels", "consume strided quantization inputs", the
suite's axis / non-contiguous / padding tests, and the review excerpt that
stores the exponent byte at the block record's start)."""
import math

import numpy as np
import pytest

import oracle
from mx_block_quantization_gb300 import workloads as W


def _snr(x, y):
    x = x.astype(np.float64)
    y = y.astype(np.float64)
    return 10 * math.log10(float((x * x).sum()) / float(((x - y) ** 2).sum()))


def test_mx9_record_is_exponent_prime_then_q_of_the_split_form():
    """The packed MX9 record holds the split form's bytes: exponent first (the
    review excerpt stores it at the record start), prime, then the 16 q."""
    x = W.mx9_outliers(64, 256, seed=1)
    rec = oracle.mx_pack(x, oracle.MX9)
    q, e, p = oracle.mx9_pack(x)
    assert rec.shape == (q.shape[0], 18)
    np.testing.assert_array_equal(rec[:, 0], e)
    np.testing.assert_array_equal(rec[:, 1], p[:, 0])
    np.testing.assert_array_equal(rec[:, 2:].view(np.int8), q)
    y = oracle.mx_unpack(rec, oracle.MX9, 64, 256, "f32")
    np.testing.assert_array_equal(y, oracle.mx9_unpack(q, e, p, "f32", 64, 256))


@pytest.mark.parametrize("fmt", [oracle.MX9, oracle.MX6])
def test_bits_per_element(fmt):
    """9 bits per element for MX9 (Summary); 6 for MX6 (the format's name)."""
    assert 8 * oracle.RECORD_BYTES[fmt] / 16 == fmt


@pytest.mark.parametrize("fmt", [oracle.MX9, oracle.MX6])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_axis0_is_axis1_of_the_transpose(fmt, dt):
    x = W.mx9_outliers(96, 64, seed=2)
    if dt == "bf16":
        x = W.f32_to_bf16_bits(x)
    a = oracle.mx_pack(x, fmt, axis=0)
    b = oracle.mx_pack(np.ascontiguousarray(x.T), fmt, axis=1)
    np.testing.assert_array_equal(a, b)
    ya = oracle.mx_unpack(a, fmt, 96, 64, dt, axis=0)
    yb = oracle.mx_unpack(b, fmt, 64, 96, dt, axis=1)
    np.testing.assert_array_equal(ya, np.ascontiguousarray(yb.T))


@pytest.mark.parametrize("fmt", [oracle.MX9, oracle.MX6])
@pytest.mark.parametrize("axis", [0, 1])
def test_strided_input_equals_contiguous_copy(fmt, axis):
    x = W.normal_f32((48, 80), seed=3)
    wide = np.full((48, 112), np.float32(7e30))
    wide[:, :80] = x
    a = oracle.mx_pack(wide, fmt, axis=axis, cols=80)
    b = oracle.mx_pack(x, fmt, axis=axis)
    np.testing.assert_array_equal(a, b)
    fill = np.full((48, 112), np.float32(-3.0))
    y = oracle.mx_unpack(a, fmt, 48, 80, "f32", axis=axis, ld=112, fill=fill)
    assert (y[:, 80:] == -3.0).all()
    np.testing.assert_array_equal(y[:, :80], oracle.mx_unpack(b, fmt, 48, 80, "f32", axis=axis))


@pytest.mark.parametrize("fmt", [oracle.MX9, oracle.MX6])
@pytest.mark.parametrize("axis", [0, 1])
def test_partial_block_is_zero_padding(fmt, axis):
    """A partial last block packs as the zero-padded block; unpack writes only
    the real elements."""
    x = W.normal_f32((20, 37), seed=4)
    padded = np.zeros((32, 48), np.float32)
    padded[:20, :37] = x
    a = oracle.mx_pack(x, fmt, axis=axis)
    if axis == 1:
        b = oracle.mx_pack(np.ascontiguousarray(padded[:20]), fmt, axis=1)
    else:
        b = oracle.mx_pack(np.ascontiguousarray(padded[:, :37]), fmt, axis=0)
    np.testing.assert_array_equal(a, b)
    y = oracle.mx_unpack(a, fmt, 20, 37, "f32", axis=axis)
    yp = oracle.mx_unpack(b, fmt, 20 if axis == 1 else 32, 48 if axis == 1 else 37, "f32",
                          axis=axis)
    np.testing.assert_array_equal(y, yp[:20, :37])


def _t(v):
    if math.isnan(v) or math.isinf(v):
        return 128
    if v == 0 or abs(v) < 2.0 ** -126:
        return -127
    return math.frexp(v)[1] - 1


def _mx6_codes(rec):
    """Decode the sixteen 5-bit two's-complement codes of MX6 records."""
    bits = np.unpackbits(rec[:, 2:], axis=1, bitorder="little")
    codes = np.zeros((rec.shape[0], 16), np.int64)
    for i in range(16):
        for b in range(5):
            codes[:, i] |= bits[:, 5 * i + b].astype(np.int64) << b
    return np.where(codes >= 16, codes - 32, codes)


def test_mx6_nearest_grid_point_and_exponents():
    """MX6 brute force: shared exponent and prime bits from math.frexp, and each
    q the integer in [-15, 15] whose q*2^k is nearest (ties to even), k =
    max(E - 3 - prime, -126)."""
    g = np.random.Generator(np.random.PCG64(5))
    x = (g.standard_normal((32, 64)) * np.exp2(g.integers(-130, 100, (32, 1)))).astype(np.float32)
    rec = oracle.mx_pack(x, oracle.MX6)
    q = _mx6_codes(rec)
    grid = np.arange(-15, 16)
    blocks = x.reshape(-1, 16).astype(np.float64)
    for b in range(blocks.shape[0]):
        t = [_t(float(v)) for v in blocks[b]]
        E = max(t)
        assert rec[b, 0] == E + 127
        for i in range(16):
            tau = int(max(t[2 * (i // 2)], t[2 * (i // 2) + 1]) < E)
            assert (rec[b, 1] >> (i // 2)) & 1 == tau
            k = max(E - 3 - tau, -126)
            d = np.abs(grid * 2.0 ** k - blocks[b, i])
            best = grid[d == d.min()]
            want = best[0] if best.size == 1 else best[best % 2 == 0][0]
            assert q[b, i] == want


def test_mx6_loses_about_three_bits_against_mx9():
    """Three fewer magnitude bits cost about 6.02 dB each on Gaussian data."""
    x = W.normal_f32((512, 512), seed=6)
    y9 = oracle.mx_unpack(oracle.mx_pack(x, oracle.MX9), oracle.MX9, 512, 512, "f32")
    y6 = oracle.mx_unpack(oracle.mx_pack(x, oracle.MX6), oracle.MX6, 512, 512, "f32")
    d = _snr(x, y9) - _snr(x, y6)
    assert 16.0 <= d <= 20.0, d
    assert _snr(x, y6) > 25.0


@pytest.mark.parametrize("fmt", [oracle.MX9, oracle.MX6])
def test_idempotent_and_symmetric(fmt):
    x = W.mx9_outliers(64, 128, seed=7)
    a = oracle.mx_pack(x, fmt)
    y = oracle.mx_unpack(a, fmt, 64, 128, "f32")
    np.testing.assert_array_equal(oracle.mx_pack(y, fmt), a)
    neg = oracle.mx_pack(-x, fmt)
    np.testing.assert_array_equal(neg[:, :2], a[:, :2])
    if fmt == oracle.MX9:
        np.testing.assert_array_equal(neg[:, 2:].view(np.int8), -a[:, 2:].view(np.int8))
    else:
        np.testing.assert_array_equal(_mx6_codes(neg), -_mx6_codes(a))


def test_every_mx6_code_round_trips():
    """Pairs (15, q) for every q in [-15, 15]: each pair holds an element of the
    block exponent E = 3, so no pair is demoted, k = 0, and the codes are the
    values themselves; unpack returns the input exactly."""
    qs = np.arange(-15, 16)
    pairs = np.stack([np.full_like(qs, 15), qs], axis=1).reshape(-1).astype(np.float32)
    x = np.zeros(64, np.float32)
    x[:pairs.size] = pairs
    x[pairs.size:] = 15.0
    x = x.reshape(4, 16)
    rec = oracle.mx_pack(x, oracle.MX6)
    assert (rec[:, 0] == 3 + 127).all() and (rec[:, 1] == 0).all()
    codes = _mx6_codes(rec).reshape(-1)
    np.testing.assert_array_equal(codes[1:pairs.size:2], qs)
    np.testing.assert_array_equal(oracle.mx_unpack(rec, oracle.MX6, 4, 16, "f32"), x)


@pytest.mark.parametrize("fmt,off,qmax", [(oracle.MX9, 6, 127), (oracle.MX6, 3, 15)])
@pytest.mark.parametrize("bf16", [False, True])
def test_brute_force_at_the_exponent_floor(fmt, off, qmax, bf16):
    """Blocks of zeros, subnormals and the smallest normals (every largest field
    <= 8), where k = max(E - off - prime, -126) sits at or near its floor and a
    subnormal rounds to 0 or +-1: exponent byte, prime bits and each q as the
    nearest grid point (ties to even), from math.frexp on the exact input; the
    unpack returns q * 2^k exactly (|q| * 2^k is 0 or at least 2^-126)."""
    x = W.tiny_exponents(32, 64, bf16, seed=17 + fmt)
    v = W.bf16_bits_to_f32(x) if bf16 else x
    rec = oracle.mx_pack(x, fmt)
    y = oracle.mx_unpack(rec, fmt, 32, 64, "f32").reshape(-1, 16).astype(np.float64)
    q = _mx6_codes(rec) if fmt == oracle.MX6 else rec[:, 2:].view(np.int8).astype(np.int64)
    grid = np.arange(-qmax, qmax + 1)
    blocks = v.reshape(-1, 16).astype(np.float64)
    floor_hits = 0
    for b in range(blocks.shape[0]):
        t = [_t(float(e)) for e in blocks[b]]
        E = max(t)
        assert rec[b, 0] == E + 127
        for i in range(16):
            tau = int(max(t[2 * (i // 2)], t[2 * (i // 2) + 1]) < E)
            assert (rec[b, 1] >> (i // 2)) & 1 == tau
            k = max(E - off - tau, -126)
            floor_hits += k == -126
            d = np.abs(grid * 2.0 ** k - blocks[b, i])
            best = grid[d == d.min()]
            want = best[0] if best.size == 1 else best[best % 2 == 0][0]
            assert q[b, i] == want, (b, i, blocks[b, i], k)
            assert y[b, i] == want * 2.0 ** k, (b, i, y[b, i], k)
    assert floor_hits > 100
