"""A second, independent statement of the whole dual-axis MXFP8 cast, for small
inputs, and the C oracle held to it byte for byte.

The twin shares nothing with the oracle: NumPy for the blocks, the scale byte
as the smallest s in [0, 254] with amax <= 448 * 2^(s - 127) found by search
(pytorch/ao PR #4995, "Fused dual-axis MXFP8 quantization with correct
metadata": the rceil rule, the printed cutoff, the non-finite list and the NaN
paragraph), PyTorch's float8_e4m3fn cast for the data bytes (OCP E4M3, round to
nearest even, a library routine), the 128x4 blocked layout as a reshape and
permute, and the colwise scales as contiguous per-group slabs with the
uncovered tail zeroed (the "Uncovered tail" paragraph).  A slip anywhere in the
oracle's dual path (an index, a stride, a rule, a slab offset) breaks equality.
"""
import numpy as np
import pytest
import torch

import oracle
from mx_block_quantization_gb300 import workloads as W


def _scale(amax: float) -> int:
    s = 0
    while s < 254 and amax > 448.0 * 2.0 ** (s - 127):
        s += 1
    return s


def _e4m3(v: np.ndarray) -> np.ndarray:
    """|v| <= 448 (or +-Inf, saturated to +-448) -> E4M3 bytes, sign kept (-0 -> 0x80)."""
    v = np.where(np.isinf(v), np.copysign(448.0, v), v)
    return torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _blocks(lines: np.ndarray, colwise: bool):
    """lines: [L, K] float64, blocks of 32 along K -> (scales [L, K/32], codes [L, K])."""
    L, K = lines.shape
    s = np.zeros((L, K // 32), np.uint8)
    q = np.zeros((L, K), np.uint8)
    for i in range(L):
        for j in range(K // 32):
            b = lines[i, 32 * j:32 * j + 32]
            if np.isnan(b).any() or (np.isinf(b).any() and not colwise):
                s[i, j] = 255                       # all-NaN block
                q[i, 32 * j:32 * j + 32] = 0x7F
                continue
            sc = 254 if np.isinf(b).any() else _scale(float(np.abs(b).max()))
            s[i, j] = sc
            q[i, 32 * j:32 * j + 32] = _e4m3(b * 2.0 ** (127 - sc))
    return s, q


def _blocked(S: np.ndarray) -> np.ndarray:
    """[R, C] scales (R % 128 == 0, C % 4 == 0) -> the 128x4 blocked byte order."""
    R, C = S.shape
    return S.reshape(R // 128, 4, 32, C // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)


def twin_dual(x_bits: np.ndarray, offs):
    M, N = x_bits.shape
    with np.errstate(invalid="ignore"):  # NaN payloads
        x = W.bf16_bits_to_f32(x_bits).astype(np.float64)
    s_r, q_r = _blocks(x, colwise=False)
    s_c, q_c = _blocks(np.ascontiguousarray(x.T), colwise=True)   # [N, M/32], [N, M]
    bounds = [M] if offs is None else [int(o) for o in offs]
    s_col = np.zeros(N * M // 32, np.uint8)
    lo = 0
    for hi in bounds:
        if hi > lo:
            s_col[N * lo // 32:N * hi // 32] = _blocked(s_c[:, lo // 32:hi // 32])
        lo = hi
    return {"q_row": q_r.reshape(-1), "s_row": _blocked(s_r), "q_col": q_c.reshape(-1),
            "s_col": s_col}


def _specials(M, N, seed):
    """Scaled normals per 32-row band, zero and subnormal blocks, +-Inf, NaN, -0,
    the printed cutoff's neighbours and the largest finite bf16."""
    x = W.dual_specials(M, N, seed=seed)
    g = np.random.Generator(np.random.PCG64(seed))
    x[32:64, 64:96] = 0                                       # a zero 32x32 block
    x[64:96, 32:64] = (g.integers(1, 128, (32, 32)) | (g.integers(0, 2, (32, 32)) << 15)).astype(np.uint16)
    r, c = g.integers(96, M, 12), g.integers(0, N, 12)        # (subnormals only above)
    x[r[0], c[0]] = 0x8000                                    # -0
    x[r[1], c[1]] = 0x0460                                    # cutoff: scale 0
    x[r[2], c[2]] = 0x0461                                    # above it: scale 1
    x[r[3], c[3]] = 0x7F7F                                    # largest finite
    x[r[4], c[4]] = 0xFF80                                    # -Inf
    x[r[5], c[5]] = 0x7FC1                                    # NaN with payload
    return x


CASES = [
    ("small N(0,1), one group", lambda: W.dual_small()),
    ("specials 256x256 dense", lambda: (_specials(256, 256, 1), None)),
    ("specials 384x256, empty group and tail", lambda: (_specials(384, 256, 2),
                                                       np.array([128, 128, 256], np.int32))),
    ("specials 512x128, four groups", lambda: (_specials(512, 128, 3),
                                              np.array([0, 256, 384, 512], np.int32))),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_oracle_equals_independent_twin(name, make):
    x, offs = make()
    want = twin_dual(x, offs)
    got = oracle.mxfp8_dual(x, offs)
    for k in ("q_row", "s_row", "q_col", "s_col"):
        bad = np.flatnonzero(got[k] != want[k])
        assert bad.size == 0, (f"{name}: {k} differs at {bad[:8]} "
                               f"(got {got[k][bad[:4]]}, twin {want[k][bad[:4]]})")


def test_twin_sees_every_rule():
    """The special cases reach every branch of the twin: NaN and Inf blocks both
    ways, scale 0, the largest finite scale, subnormal-only blocks."""
    x, offs = _specials(384, 256, 2), np.array([128, 128, 256], np.int32)
    t = twin_dual(x, offs)
    assert (t["s_row"] == 255).any() and (t["s_col"] == 255).any() and (t["s_col"] == 254).any()
    assert (t["s_row"] == 0).any() and (t["s_row"] == 247).any()
    assert (t["s_col"][256 * 256 // 32:] == 0).all()        # the tail rows 256..383
    assert (t["q_row"].reshape(384, 256)[64:96, 32:64] != 0).any()  # subnormals scaled up
