"""Seeded synthetic inputs shaped like the published workloads.

Every generator draws from numpy's PCG64 with an explicit seed, builds the
tensor on the host and returns plain numpy arrays (bf16 tensors as uint16 bit
patterns), so the GPU path and the CPU oracle consume identical bytes.  This
module holds no quantization arithmetic: only random draws, the fp32 -> bf16
round-to-nearest-even used to make bf16 inputs, and the placement of special
values.

Workloads (shapes and recipes as published for this method; the pages use no
public dataset):

* ``dual_small``      -- 128 x 128 bf16 N(0,1), one group (offs = [128]).
* ``mx9_outliers``    -- [4096, 4096] N(0,1), 1% of elements x100, 64 all-zero
  16-blocks and 64 16-blocks of magnitude ~1e-40 (fp32 subnormal); the bf16
  variant is the same tensor rounded to bf16.
* ``dual_specials``   -- 8192 x 8192 bf16 N(0,1) x 2^u per 32-row band, u an
  integer uniform in [-30, 15]; 1% of the 32x32 blocks zeroed (half) or filled
  with random-sign bf16 subnormals (half); then 0.01% of elements +-Inf and
  0.01% NaN at distinct positions.
* ``moe_grouped``     -- [65536, 7168] bf16 N(0,1) * 0.02, 64 expert groups of
  128 * Multinomial(448, 1/64) rows: offs[-1] = 57344, an 8192-row uncovered
  tail; some groups can be empty.
* ``tiny_exponents``  -- blocks at the scale exponent's floor: zeros,
  subnormals and the smallest normals (exponent field <= a per-16x16-tile cap
  in 0..8), fp32 or bf16 bit patterns.
* ``SWEEP_SHAPES``    -- throughput sweep shapes, N(0,1).
"""
from __future__ import annotations

import numpy as np

SEED = 0

SWEEP_SHAPES = [(1024, 1024), (4096, 4096), (16384, 8192), (32768, 16384)]


def rng(seed: int = SEED) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); NaN -> 0x7FC0 | sign."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint32(16)) & np.uint32(0x8000)).astype(np.uint16) | np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_f32(shape, seed: int = SEED, scale: float = 1.0) -> np.ndarray:
    x = rng(seed).standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def normal_bf16(shape, seed: int = SEED, scale: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits(normal_f32(shape, seed, scale))


# ---------------------------------------------------------------------------
# dual-axis MXFP8 workloads
# ---------------------------------------------------------------------------

def dual_small(seed: int = SEED) -> tuple[np.ndarray, np.ndarray]:
    """128 x 128 bf16 N(0,1) and offs = [128]."""
    return normal_bf16((128, 128), seed), np.array([128], dtype=np.int32)


def dual_specials(M: int = 8192, N: int = 8192, seed: int = SEED) -> np.ndarray:
    """Dense bf16 tensor exercising scale bytes 0, 254 and 255 (see module doc)."""
    g = rng(seed)
    x = g.standard_normal(size=(M, N), dtype=np.float32)
    u = g.integers(-30, 16, size=M // 32)                      # per 32-row band
    x *= np.repeat(np.exp2(u).astype(np.float32), 32)[:, None]
    b = f32_to_bf16_bits(x)
    # 1% of the 32x32 blocks: half zero, half random-sign subnormals
    nblk = (M // 32) * (N // 32)
    nsel = nblk // 100
    sel = g.choice(nblk, size=nsel, replace=False)
    bv = b.reshape(M // 32, 32, N // 32, 32)
    for k, blk in enumerate(sel):
        bi, bj = divmod(int(blk), N // 32)
        if k < nsel // 2:
            bv[bi, :, bj, :] = 0
        else:
            mant = g.integers(1, 128, size=(32, 32), dtype=np.uint16)
            sign = g.integers(0, 2, size=(32, 32), dtype=np.uint16) << np.uint16(15)
            bv[bi, :, bj, :] = sign | mant
    # 0.01% +-Inf, then 0.01% NaN (random sign and payload), distinct positions
    nspec = int(round(M * N * 1e-4))
    pos = g.choice(M * N, size=2 * nspec, replace=False)
    flat = b.reshape(-1)
    inf_sign = g.integers(0, 2, size=nspec, dtype=np.uint16) << np.uint16(15)
    flat[pos[:nspec]] = inf_sign | np.uint16(0x7F80)
    nan_sign = g.integers(0, 2, size=nspec, dtype=np.uint16) << np.uint16(15)
    nan_mant = g.integers(1, 128, size=nspec, dtype=np.uint16)
    flat[pos[nspec:]] = nan_sign | np.uint16(0x7F80) | nan_mant
    return b


def moe_group_offsets(experts: int = 64, routed_units: int = 448, unit: int = 128,
                      seed: int = SEED) -> np.ndarray:
    """Cumulative group ends: sizes = unit * Multinomial(routed_units, 1/experts)."""
    counts = rng(seed).multinomial(routed_units, [1.0 / experts] * experts)
    return (np.cumsum(counts) * unit).astype(np.int32)


def moe_grouped(M: int = 65536, N: int = 7168, experts: int = 64, routed_units: int = 448,
                seed: int = SEED) -> tuple[np.ndarray, np.ndarray]:
    """bf16 [M, N] N(0,1)*0.02 and the K-group offsets (offs[-1] = 128*routed_units)."""
    offs = moe_group_offsets(experts, routed_units, 128, seed + 1)
    return normal_bf16((M, N), seed, 0.02), offs


# ---------------------------------------------------------------------------
# MX9 workloads
# ---------------------------------------------------------------------------

def mx9_outliers(rows: int = 4096, cols: int = 4096, seed: int = SEED,
                 outlier_frac: float = 0.01, outlier_mult: float = 100.0,
                 zero_blocks: int = 64, tiny_blocks: int = 64) -> np.ndarray:
    """float32 [rows, cols]: N(0,1), outliers, all-zero and ~1e-40 16-blocks."""
    g = rng(seed)
    x = g.standard_normal(size=(rows, cols), dtype=np.float32)
    flat = x.reshape(-1)
    n_out = int(round(flat.size * outlier_frac))
    if n_out:
        flat[g.choice(flat.size, size=n_out, replace=False)] *= np.float32(outlier_mult)
    nb = flat.size // 16                                            # whole 16-blocks
    blocks = g.choice(nb, size=zero_blocks + tiny_blocks, replace=False)
    bv = flat[:nb * 16].reshape(nb, 16)
    bv[blocks[:zero_blocks]] = 0.0
    tiny = g.standard_normal(size=(tiny_blocks, 16)) * 1e-40       # float64, then
    bv[blocks[zero_blocks:]] = tiny.astype(np.float32)              # fp32 subnormals
    return x


def mx9_outliers_bf16(rows: int = 4096, cols: int = 4096, seed: int = SEED) -> np.ndarray:
    return f32_to_bf16_bits(mx9_outliers(rows, cols, seed))


def tiny_exponents(rows: int, cols: int, bf16: bool, seed: int = SEED) -> np.ndarray:
    """Every element zero, subnormal or a normal with exponent field 1..cap,
    random sign and mantissa, cap drawn from 0..8 per 16x16 tile (0: subnormals
    only), so that every 16-block along either axis has its largest field at 8
    or below; 10% of mantissas sit at exactly half of their step's range (bf16
    0x40, fp32 1 << 22).  fp32 as float32, bf16 as uint16 bit patterns."""
    g = rng(seed)
    cap = np.repeat(np.repeat(g.integers(0, 9, (rows // 16 + 1, cols // 16 + 1)), 16, 0), 16, 1)
    cap = cap[:rows, :cols]
    normal = (g.random((rows, cols)) >= 0.6) & (cap > 0)
    field = np.where(normal, 1 + (g.random((rows, cols)) * np.maximum(cap, 1)).astype(np.int64), 0)
    sign = g.integers(0, 2, (rows, cols))
    if bf16:
        mant = g.integers(0, 128, (rows, cols))
        mant[g.random((rows, cols)) < 0.1] = 64
        return ((sign << 15) | (field << 7) | mant).astype(np.uint16)
    mant = g.integers(0, 1 << 23, (rows, cols))
    mant[g.random((rows, cols)) < 0.1] = 1 << 22
    return ((sign << 31) | (field << 23) | mant).astype(np.uint32).view(np.float32)
