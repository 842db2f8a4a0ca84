"""The seeded input generators produce the published workload recipes, deterministically."""
import numpy as np
import pytest

from mx_block_quantization_gb300 import workloads as W


def test_bf16_rounding_is_nearest_even():
    import torch
    g = np.random.Generator(np.random.PCG64(1))
    x = (g.standard_normal(100000) * np.exp2(g.integers(-140, 120, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(W.f32_to_bf16_bits(x), ref)


def test_deterministic():
    a = W.dual_specials(256, 256, seed=0)
    b = W.dual_specials(256, 256, seed=0)
    assert np.array_equal(a, b)
    assert np.array_equal(W.mx9_outliers(64, 64), W.mx9_outliers(64, 64))


def test_moe_offsets_recipe():
    offs = W.moe_group_offsets()
    assert offs.dtype == np.int32 and offs.size == 64
    assert offs[-1] == 57344 and np.all(np.diff(np.r_[0, offs]) >= 0)
    assert np.all(offs % 128 == 0)


def test_specials_recipe_counts():
    M = N = 1024
    x = W.dual_specials(M, N)
    v = W.bf16_bits_to_f32(x)
    nspec = int(round(M * N * 1e-4))
    assert np.isinf(v).sum() == nspec and np.isnan(v).sum() == nspec
    sub = (x & 0x7F80) == 0
    # half of 1% of the 32x32 blocks hold random-sign subnormals (a few may be
    # overwritten by the Inf/NaN placed afterwards)
    n_sub_blocks = (M // 32) * (N // 32) // 100 - (M // 32) * (N // 32) // 100 // 2
    assert ((x & 0x7FFF) != 0)[sub].sum() >= 0.98 * 32 * 32 * n_sub_blocks


def test_mx9_recipe_counts():
    x = W.mx9_outliers(512, 512)
    blocks = x.reshape(-1, 16)
    assert (np.abs(blocks).max(axis=1) == 0).sum() >= 64
    tiny = (np.abs(blocks).max(axis=1) > 0) & (np.abs(blocks).max(axis=1) < 1e-37)
    assert tiny.sum() == 64
    assert (np.abs(x) > 20).mean() > 0.005


@pytest.mark.parametrize("bf16", [False, True])
def test_tiny_exponents_recipe(bf16):
    x = W.tiny_exponents(256, 320, bf16, seed=3)
    assert np.array_equal(x.view(np.uint8), W.tiny_exponents(256, 320, bf16, seed=3).view(np.uint8))
    bits = x.astype(np.uint32) if bf16 else x.view(np.uint32)
    field = (bits >> 7) & 0xFF if bf16 else (bits >> 23) & 0xFF
    assert field.max() <= 8
    tiles = field.reshape(16, 16, 20, 16).max(axis=(1, 3))   # largest field per 16x16 tile
    assert (tiles == 0).any() and (tiles == 8).any()          # subnormal-only tiles and the cap
    half = 0x40 if bf16 else 1 << 22
    mant = bits & (0x7F if bf16 else 0x7FFFFF)
    assert 0.08 < (mant == half).mean() < 0.14
    assert 0.5 < (field == 0).mean() < 0.8
