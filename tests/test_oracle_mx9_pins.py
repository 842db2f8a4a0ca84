"""Pins of the CPU oracle's MX9 half against facts that do not come from the oracle.

Source: AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with
pack/unpack" (Summary, "Key design choices", test plan, the test excerpt and the
review thread).  Each test names the mistake it catches.
"""
import math

import numpy as np
import pytest

import oracle
from mx_block_quantization_gb300 import workloads as W
from tests.conftest import golden_path


def _facts():
    out = {}
    with open(golden_path("mx9_page_facts.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


FACTS = _facts()


def _snr_db(x, y):
    x = x.astype(np.float64)
    y = y.astype(np.float64)
    return 10.0 * math.log10(float((x * x).sum()) / float(((x - y) ** 2).sum()))


def _t_frexp(v: float) -> int:
    """Element exponent from the math library: floor(log2|v|) for normal values,
    -127 for zero and fp32 subnormals, 128 for Inf/NaN."""
    if math.isnan(v) or math.isinf(v):
        return 128
    if v == 0.0 or abs(v) < 2.0 ** -126:
        return -127
    return math.frexp(v)[1] - 1


def _k(E, tau):
    return max(E - 6 - tau, -126)


# ---------------------------------------------------------------------------

def test_storage_is_nine_bits_per_element():
    """Summary: q [n_blocks,16] int8 + max_exp [n_blocks] + prime [n_blocks,1] = 9 bits/elem."""
    x = W.normal_f32((64, 256), seed=1)
    q, e, p = oracle.mx9_pack(x)
    assert q.shape == (64 * 256 // 16, 16) and q.dtype == np.int8
    assert e.shape == (64 * 256 // 16,) and e.dtype == np.uint8
    assert p.shape == (64 * 256 // 16, 1) and p.dtype == np.uint8
    bits = 8 * (q.nbytes + e.nbytes + p.nbytes) / x.size
    assert bits == FACTS["bits_per_element"]
    assert q.shape[1] == FACTS["block_size"]


def test_snr_matches_page():
    """Test plan: ~46 dB clean, ~42 dB with outliers (floors 25/15).

    Catches: dropping the prime bit (gives about 42.8/37.9 dB), a scale offset
    other than 6 (loses 6 dB per bit or saturates), truncation for rounding.
    """
    clean = W.normal_f32((1024, 1024), seed=0)
    outl = W.mx9_outliers(1024, 1024, seed=0)
    for x, want, floor in ((clean, FACTS["snr_clean_db"], FACTS["snr_clean_floor_db"]),
                           (outl, FACTS["snr_outlier_db"], FACTS["snr_outlier_floor_db"])):
        q, e, p = oracle.mx9_pack(x)
        y = oracle.mx9_unpack(q, e, p, "f32", *x.shape)
        s = _snr_db(x, y)
        assert s > floor
        assert abs(s - want) <= 1.0, s


def test_demoted_128_fraction_matches_page():
    """Key design choices: the +-127 clamp bites at the demoted +-128 boundary for
    about 0.1% of elements.  Catches: clamping to +-128, a wrong demotion rule."""
    x = W.normal_f32((1024, 1024), seed=0)
    q, e, p = oracle.mx9_pack(x)
    E = e.astype(np.int64) - 127
    tau = np.repeat((p[:, 0:1] >> np.arange(8)[None, :]) & 1, 2, axis=1)
    k = np.maximum(E[:, None] - 6 - tau, -126)
    r = np.rint(x.reshape(-1, 16).astype(np.float64) / np.exp2(k))
    frac = float(((np.abs(r) >= 128) & (tau == 1)).mean())
    assert 0.5 * FACTS["demoted_128_fraction"] <= frac <= 2.0 * FACTS["demoted_128_fraction"]
    assert np.abs(q.astype(np.int64)).max() == 127
    assert np.all(q[np.abs(r) >= 128] == np.sign(r[np.abs(r) >= 128]) * 127)


def test_max_exp_range_on_random_fp32():
    """Test excerpt: random fp32 keeps the biased shared exponent in [1, 254]."""
    x = (W.normal_f32((16, 64), seed=4))
    _, e, _ = oracle.mx9_pack(x)
    assert e.min() >= FACTS["max_exp_min"] and e.max() <= FACTS["max_exp_max"]
    g = np.random.Generator(np.random.PCG64(9))
    x = (g.standard_normal((64, 64)) * np.exp2(g.integers(-120, 120, (64, 64)))).astype(np.float32)
    _, e, _ = oracle.mx9_pack(x)
    assert e.min() >= 1 and e.max() <= 254


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shared_exponent_and_prime_against_frexp(dtype):
    """max_exp and the prime bits equal what math.frexp gives element by element.

    Catches: exponent taken from the wrong bits (bf16 bits 14..7), a wrong bias,
    a flipped prime polarity, a pair index off by one.
    """
    g = np.random.Generator(np.random.PCG64(21))
    x = (g.standard_normal((256, 64)) * np.exp2(g.integers(-135, 120, (256, 64)))).astype(np.float32)
    x[0, :16] = 0
    x[1, :16] = np.float32(1e-40)
    x[2, 5] = np.inf
    x[3, 0] = np.nan
    if dtype == "bf16":
        xin = W.f32_to_bf16_bits(x)
        xv = W.bf16_bits_to_f32(xin).astype(np.float64)
    else:
        xin = x
        xv = x.astype(np.float64)
    _, e, p = oracle.mx9_pack(xin)
    for b in range(xv.size // 16):
        blk = xv.reshape(-1, 16)[b]
        t = [_t_frexp(float(v)) for v in blk]
        E = max(t)
        assert e[b] == E + 127, b
        want = 0
        for pr in range(8):
            if max(t[2 * pr], t[2 * pr + 1]) < E:
                want |= 1 << pr
        assert p[b, 0] == want, b


def test_q_is_nearest_point_of_the_pair_grid():
    """Brute force: each q is the integer in [-127, 127] whose q*2^k_p is nearest
    to x (ties to the even q), k_p from the block exponent and the prime bit.

    Catches: truncation, ties away from zero, a clamp to +-128, k_p off by one.
    """
    g = np.random.Generator(np.random.PCG64(5))
    x = (g.standard_normal((64, 64)) * np.exp2(g.integers(-130, 100, (64, 1)))).astype(np.float32)
    # exact ties: values at (n + 1/2) * 2^k for a block with a known exponent
    x[0, :16] = np.float32(1.0)
    x[0, 2] = np.float32(1.0 + 2.0 ** -7)        # tie between 64 and 65 steps of 2^-6
    x[0, 4] = np.float32(1.0 + 3 * 2.0 ** -7)    # tie between 65 and 66
    q, e, p = oracle.mx9_pack(x)
    grid = np.arange(-127, 128)
    for b in range(x.size // 16):
        E = int(e[b]) - 127
        for i in range(16):
            tau = (int(p[b, 0]) >> (i // 2)) & 1
            k = _k(E, tau)
            v = float(x.reshape(-1, 16)[b, i])
            d = np.abs(grid * 2.0 ** k - v)
            best = grid[d == d.min()]
            want = best[0] if best.size == 1 else best[best % 2 == 0][0]
            assert q[b, i] == want, (b, i, v, q[b, i], want)
    assert q[0, 2] == 64 and q[0, 4] == 66


def test_zero_and_subnormal_blocks():
    """Zero blocks: max_exp 0, prime 0, q 0.  ~1e-40 blocks: the -126 clamp gives
    q = 0 (the scale exponent never goes below the fp32 normal range)."""
    x = np.zeros((2, 16), np.float32)
    x[1] = np.float32(1e-40) * np.arange(1, 17, dtype=np.float32)
    q, e, p = oracle.mx9_pack(x)
    assert e.tolist() == [0, 0] and p[:, 0].tolist() == [0, 0]
    assert not q.any()
    # a subnormal large enough to reach half a step of 2^-126 rounds to +-1
    y = np.zeros((1, 16), np.float32)
    y[0, 0] = np.float32(0.75 * 2.0 ** -126)
    y[0, 1] = np.float32(-0.75 * 2.0 ** -126)
    q, e, _ = oracle.mx9_pack(y)
    assert e[0] == 0 and q[0, 0] == 1 and q[0, 1] == -1


def test_pack_unpack_pack_idempotent_and_unpack_exact():
    """unpack is exactly q*2^k; pack(unpack(pack x)) == pack x byte for byte."""
    x = W.mx9_outliers(256, 256, seed=3)
    q, e, p = oracle.mx9_pack(x)
    y = oracle.mx9_unpack(q, e, p, "f32", 256, 256)
    yb = y.reshape(-1, 16)
    for b in range(0, yb.shape[0], 17):
        E = int(e[b]) - 127
        for i in range(16):
            tau = (int(p[b, 0]) >> (i // 2)) & 1
            assert float(yb[b, i]) == math.ldexp(float(q[b, i]), _k(E, tau))
    q2, e2, p2 = oracle.mx9_pack(y)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(e2, e)
    np.testing.assert_array_equal(p2, p)


def test_negation_symmetry():
    """Layer 3 of the page's suite: negating x negates q, keeps max_exp and prime."""
    x = W.mx9_outliers(128, 256, seed=8)
    a = oracle.mx9_pack(x)
    b = oracle.mx9_pack(-x)
    np.testing.assert_array_equal(b[0], -a[0])
    np.testing.assert_array_equal(b[1], a[1])
    np.testing.assert_array_equal(b[2], a[2])


def test_bf16_input_equals_its_fp32_widening():
    """A bf16 tensor and its exact fp32 widening pack identically."""
    xb = W.mx9_outliers_bf16(128, 128, seed=2)
    a = oracle.mx9_pack(xb)
    b = oracle.mx9_pack(W.bf16_bits_to_f32(xb))
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_unpack_bf16_equals_fp32_rounded():
    x = W.mx9_outliers(128, 128, seed=6)
    q, e, p = oracle.mx9_pack(x)
    yf = oracle.mx9_unpack(q, e, p, "f32", 128, 128)
    yb = oracle.mx9_unpack(q, e, p, "bf16", 128, 128)
    np.testing.assert_array_equal(yb, W.f32_to_bf16_bits(yf))
    np.testing.assert_array_equal(W.bf16_bits_to_f32(yb), yf)  # exact in bf16


def test_nonfinite_reading():
    """Reading for non-finite input (the page leaves it open): the block exponent
    is 255, NaN packs to 0, +-Inf to +-127, and unpack gives back +-Inf."""
    x = np.ones((1, 16), np.float32)
    x[0, 0] = np.inf
    x[0, 1] = -np.inf
    x[0, 2] = np.nan
    q, e, p = oracle.mx9_pack(x)
    assert e[0] == 255
    assert q[0, 0] == 127 and q[0, 1] == -127 and q[0, 2] == 0
    y = oracle.mx9_unpack(q, e, p, "f32", 1, 16)
    assert y[0, 0] == np.inf and y[0, 1] == -np.inf


def test_bad_arguments_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.mx9_pack(np.zeros((4, 15), np.float32))
    with pytest.raises(TypeError):
        oracle.mx9_pack(np.zeros((4, 16), np.float16))
