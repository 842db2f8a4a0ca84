"""CPU oracle for MX block quantization -- TEST INFRASTRUCTURE.

A plain, slow, scalar C implementation (``mxq_oracle.c``) of what the GPU
library computes, written from the published definitions:

* pytorch/ao PR #4995 "Fused dual-axis MXFP8 quantization with correct
  metadata" (description and review replies): 1x32 / 32x1 MXFP8 blocks, rceil
  E8M0 scales, the non-finite rules, blocked scales, K-group slabs and the
  zeroed uncovered tail.
* AMD-AGI/ALTO PR #33 "mx9: add fused MX9 quantization kernel with pack/unpack"
  (Summary, "Key design choices", review thread): MX9 pack/unpack.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does, and this
package imports nothing from the product.

This module only marshals numpy arrays into the C functions; every step of
the arithmetic is in the C file.

Parity unpinned (not printed on the pages): the bit order of the MX9 / MX6
prime byte, the sign of the E4M3 NaN byte and the MX6 5-bit code layout.
Every other result has at least one pin outside the oracle.
"""
from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SRC = _HERE / "mxq_oracle.c"
_LIB = _HERE / "libmxq_oracle.so"
# A prebuilt oracle library to load instead (the mutation test points this at
# deliberately broken copies to show that the pins catch them).
_LIB_OVERRIDE = os.environ.get("MXQ_ORACLE_LIB")

F32 = 0
BF16 = 1

OK = 0
EBADSHAPE = -1
EBADDTYPE = -2
EBADOFFS = -3


def build(force: bool = False) -> pathlib.Path:
    """Compile the oracle with gcc (strict IEEE: no fast-math, no FMA contraction)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_name(f".{_LIB.name}.{os.getpid()}.tmp")
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-frounding-math", "-Wall", "-Wextra",
             str(_SRC), "-o", str(tmp), "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(_LIB_OVERRIDE if _LIB_OVERRIDE else str(build()))
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e8m0_rceil.restype = ctypes.c_int
        lib.oracle_e8m0_rceil.argtypes = [ctypes.c_double]
        lib.oracle_blocked_index.restype = i64
        lib.oracle_blocked_index.argtypes = [i64, i64, i64, i64]
        lib.oracle_mxfp8_block.restype = None
        lib.oracle_mxfp8_block.argtypes = [p, i64, ctypes.c_int, p, p, i64]
        lib.oracle_check_offs.restype = ctypes.c_int
        lib.oracle_check_offs.argtypes = [p, ctypes.c_int32, i64]
        lib.oracle_mxfp8_dual.restype = ctypes.c_int
        lib.oracle_mxfp8_dual.argtypes = [p, i64, i64, p, ctypes.c_int32, p, p, p, p]
        lib.oracle_mx9_pack.restype = ctypes.c_int
        lib.oracle_mx9_pack.argtypes = [p, ctypes.c_int, i64, i64, p, p, p]
        lib.oracle_mx9_unpack.restype = ctypes.c_int
        lib.oracle_mx9_unpack.argtypes = [p, p, p, p, ctypes.c_int, i64, i64]
        lib.oracle_mxfp8_block_nan_dropped.restype = None
        lib.oracle_mxfp8_block_nan_dropped.argtypes = [p, i64, p, p, i64]
        lib.oracle_mxfp8_1x32.restype = ctypes.c_int
        lib.oracle_mxfp8_1x32.argtypes = [p, i64, i64, p, p]
        lib.oracle_mxfp8_32x1.restype = ctypes.c_int
        lib.oracle_mxfp8_32x1.argtypes = [p, i64, i64, p, p]
        lib.oracle_swizzle_kgroups.restype = ctypes.c_int
        lib.oracle_swizzle_kgroups.argtypes = [p, i64, i64, p, ctypes.c_int32, p]
        lib.oracle_mx_pack.restype = ctypes.c_int
        lib.oracle_mx_pack.argtypes = [p, ctypes.c_int, i64, i64, i64, ctypes.c_int, ctypes.c_int, p]
        lib.oracle_mx_unpack.restype = ctypes.c_int
        lib.oracle_mx_unpack.argtypes = [p, ctypes.c_int, p, ctypes.c_int, i64, i64, i64,
                                         ctypes.c_int]
        lib.oracle_rounding_is_nearest_even.restype = ctypes.c_int
        lib.oracle_rounding_is_nearest_even.argtypes = []
        if not lib.oracle_rounding_is_nearest_even():
            raise RuntimeError("oracle needs round-to-nearest-even")
        _lib_handle = lib
    return _lib_handle


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle rejected the arguments (status {code})")
        self.code = code


# --------------------------------------------------------------------------
# scalar helpers (exposed for the pins)
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return _lib().oracle_e4m3_value(int(code))


def e4m3_encode(v: float) -> int:
    return int(_lib().oracle_e4m3_encode(float(v)))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    f = _lib().oracle_e4m3_encode
    return np.array([f(float(t)) for t in np.asarray(v, dtype=np.float64).ravel()],
                    dtype=np.uint8).reshape(np.shape(v))


def e8m0_rceil(amax: float) -> int:
    return int(_lib().oracle_e8m0_rceil(float(amax)))


def blocked_index(r: int, c: int, R: int, C: int) -> int:
    return int(_lib().oracle_blocked_index(r, c, R, C))


def mxfp8_block(values_bf16_bits: np.ndarray, colwise: bool) -> tuple[int, np.ndarray]:
    """Quantize one block of 32 bf16 bit patterns; returns (scale byte, 32 data bytes)."""
    x = np.ascontiguousarray(values_bf16_bits, dtype=np.uint16)
    assert x.size == 32
    s = np.zeros(1, np.uint8)
    q = np.zeros(32, np.uint8)
    _lib().oracle_mxfp8_block(_ptr(x), 1, int(bool(colwise)), _ptr(s), _ptr(q), 1)
    return int(s[0]), q


def mxfp8_block_nan_dropped(values_bf16_bits: np.ndarray) -> tuple[int, np.ndarray]:
    """The separate 32x1 cast's block rule (NaN skipped by the amax, Inf saturates)."""
    x = np.ascontiguousarray(values_bf16_bits, dtype=np.uint16)
    assert x.size == 32
    s = np.zeros(1, np.uint8)
    q = np.zeros(32, np.uint8)
    _lib().oracle_mxfp8_block_nan_dropped(_ptr(x), 1, _ptr(s), _ptr(q), 1)
    return int(s[0]), q


# --------------------------------------------------------------------------
# whole-tensor entry points
# --------------------------------------------------------------------------

def check_offs(offs: np.ndarray | None, M: int) -> int:
    if offs is None:
        return int(_lib().oracle_check_offs(None, 0, M))
    o = np.ascontiguousarray(offs, dtype=np.int32)
    return int(_lib().oracle_check_offs(_ptr(o), o.size, M))


def mxfp8_dual(x_bits: np.ndarray, offs: np.ndarray | None = None) -> dict[str, np.ndarray]:
    """x_bits: uint16 bf16 bit patterns [M, N].  Returns q_row, s_row, q_col, s_col (uint8, flat)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, N = x.shape
    o = None if offs is None else np.ascontiguousarray(offs, dtype=np.int32)
    G = 0 if o is None else o.size
    q_row = np.empty(M * N, np.uint8)
    q_col = np.empty(M * N, np.uint8)
    s_row = np.empty(M * N // 32, np.uint8)
    s_col = np.empty(M * N // 32, np.uint8)
    rc = _lib().oracle_mxfp8_dual(_ptr(x), M, N, _ptr(o), G, _ptr(q_row), _ptr(s_row),
                                  _ptr(q_col), _ptr(s_col))
    if rc != OK:
        raise OracleError(rc)
    return {"q_row": q_row, "s_row": s_row, "q_col": q_col, "s_col": s_col}


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    raise TypeError(f"unsupported dtype {x.dtype} (float32 or uint16 bf16 bits)")


def mx9_pack(x: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """x: float32, or uint16 bf16 bit patterns, shape [rows, cols] with cols % 16 == 0.

    Returns q int8 [n_blocks, 16], max_exp uint8 [n_blocks], prime uint8 [n_blocks, 1].
    """
    x = np.ascontiguousarray(x)
    dt = _dtype_code(x)
    rows, cols = x.shape
    nb = rows * (cols // 16)
    q = np.empty((nb, 16), np.int8)
    e = np.empty(nb, np.uint8)
    p = np.empty((nb, 1), np.uint8)
    rc = _lib().oracle_mx9_pack(_ptr(x), dt, rows, cols, _ptr(q), _ptr(e), _ptr(p))
    if rc != OK:
        raise OracleError(rc)
    return q, e, p


def mx9_unpack(q: np.ndarray, max_exp: np.ndarray, prime: np.ndarray, out_dtype: str,
               rows: int, cols: int) -> np.ndarray:
    """Rebuild [rows, cols] as float32 (out_dtype 'f32') or bf16 bit patterns ('bf16')."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    e = np.ascontiguousarray(max_exp, dtype=np.uint8)
    p = np.ascontiguousarray(prime, dtype=np.uint8)
    if out_dtype == "f32":
        dt, y = F32, np.empty((rows, cols), np.float32)
    elif out_dtype == "bf16":
        dt, y = BF16, np.empty((rows, cols), np.uint16)
    else:
        raise ValueError(out_dtype)
    rc = _lib().oracle_mx9_unpack(_ptr(q), _ptr(e), _ptr(p), _ptr(y), dt, rows, cols)
    if rc != OK:
        raise OracleError(rc)
    return y


# --------------------------------------------------------------------------
# the three-pass composition (1x32 cast, 32x1 cast, K-groups swizzle)
# --------------------------------------------------------------------------

def mxfp8_1x32(x_bits: np.ndarray) -> dict[str, np.ndarray]:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, N = x.shape
    q_row = np.empty(M * N, np.uint8)
    s_row = np.empty(M * N // 32, np.uint8)
    rc = _lib().oracle_mxfp8_1x32(_ptr(x), M, N, _ptr(q_row), _ptr(s_row))
    if rc != OK:
        raise OracleError(rc)
    return {"q_row": q_row, "s_row": s_row}


def mxfp8_32x1(x_bits: np.ndarray) -> dict[str, np.ndarray]:
    """q_col [N*M] and the plain row-major colwise scales s_rm [N, M/32]."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, N = x.shape
    q_col = np.empty(M * N, np.uint8)
    s_rm = np.empty((N, M // 32), np.uint8)
    rc = _lib().oracle_mxfp8_32x1(_ptr(x), M, N, _ptr(q_col), _ptr(s_rm))
    if rc != OK:
        raise OracleError(rc)
    return {"q_col": q_col, "s_rm": s_rm}


def swizzle_kgroups(s_rm: np.ndarray, offs: np.ndarray | None) -> np.ndarray:
    s = np.ascontiguousarray(s_rm, dtype=np.uint8)
    N, C = s.shape
    M = 32 * C
    o = None if offs is None else np.ascontiguousarray(offs, dtype=np.int32)
    out = np.empty(N * M // 32, np.uint8)
    rc = _lib().oracle_swizzle_kgroups(_ptr(s), N, M, _ptr(o), 0 if o is None else o.size, _ptr(out))
    if rc != OK:
        raise OracleError(rc)
    return out


def mxfp8_dual_3pass(x_bits: np.ndarray, offs: np.ndarray | None = None) -> dict[str, np.ndarray]:
    """What the three separate passes produce together."""
    r = mxfp8_1x32(x_bits)
    c = mxfp8_32x1(x_bits)
    return {"q_row": r["q_row"], "s_row": r["s_row"], "q_col": c["q_col"],
            "s_col": swizzle_kgroups(c["s_rm"], offs), "s_rm": c["s_rm"].reshape(-1)}


# --------------------------------------------------------------------------
# MX9 / MX6 in the single packed tensor, any axis, strided, padded
# --------------------------------------------------------------------------
MX9 = 9
MX6 = 6
RECORD_BYTES = {MX9: 18, MX6: 12}


def mx_blocks(rows: int, cols: int, axis: int) -> int:
    lines, length = (rows, cols) if axis == 1 else (cols, rows)
    return lines * ((length + 15) // 16)


def mx_pack(x: np.ndarray, fmt: int, axis: int = 1, cols: int | None = None) -> np.ndarray:
    """x: [rows, ld] float32 or bf16 bits, of which the first `cols` columns are
    the tensor (cols defaults to ld).  Returns uint8 [n_blocks, record bytes]."""
    x = np.ascontiguousarray(x)
    dt = _dtype_code(x)
    rows, ld = x.shape
    cols = ld if cols is None else cols
    out = np.zeros((mx_blocks(rows, cols, axis), RECORD_BYTES[fmt]), np.uint8)
    rc = _lib().oracle_mx_pack(_ptr(x), dt, rows, cols, ld, axis, fmt, _ptr(out))
    if rc != OK:
        raise OracleError(rc)
    return out


def mx_unpack(packed: np.ndarray, fmt: int, rows: int, cols: int, out_dtype: str,
              axis: int = 1, ld: int | None = None, fill=None) -> np.ndarray:
    """Rebuild [rows, ld] (ld defaults to cols); elements outside the tensor
    keep `fill` (a prefilled array) or zero."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    ld = cols if ld is None else ld
    if out_dtype == "f32":
        dt = F32
        y = np.zeros((rows, ld), np.float32) if fill is None else fill.copy()
    else:
        dt = BF16
        y = np.zeros((rows, ld), np.uint16) if fill is None else fill.copy()
    rc = _lib().oracle_mx_unpack(_ptr(packed), fmt, _ptr(y), dt, rows, cols, ld, axis)
    if rc != OK:
        raise OracleError(rc)
    return y
