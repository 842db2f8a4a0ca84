"""GB300-native MX block quantization: a thin Python binding over libmxq.so.

The binding only marshals torch tensors into the C ABI declared in
``include/mxq.h``; every step of the computation runs in the library's sm_103a
kernels.  There is no CPU fallback: calling an op without the built library,
or with tensors that are not on a CUDA device, raises.

Operations (sources by page title):

* :func:`quantize_2d_dual` -- pytorch/ao PR #4995 "Fused dual-axis MXFP8
  quantization with correct metadata": one read of a bf16 [M, N] tensor gives
  rowwise (1x32) and colwise (32x1) E4M3 data and both E8M0 rceil scale
  tensors in the 128x4 blocked layout, colwise scales per K-group slab with
  the tail past offs[-1] zeroed.
* :func:`mx9_pack` / :func:`mx9_unpack` -- AMD-AGI/ALTO PR #33 "mx9: add fused
  MX9 quantization kernel with pack/unpack": block 16, int8 q in [-127, 127],
  E8M0 shared exponent, one prime bit per pair.
* :func:`mx_pack_packed` / :func:`mx_unpack_packed` -- the same page's later
  commits: MX9 or MX6 records in one uint8 tensor, blocked along either axis of
  a strided tensor, a partial last block zero-padded.
* :func:`quantize_1x32`, :func:`quantize_32x1`, :func:`swizzle_kgroups`,
  :func:`quantize_2d_dual_3pass` -- the three-pass composition the fused cast
  replaces (pytorch/ao PR #4995, first paragraph), for comparison.
* :func:`mxfp8_scaled_mm` -- a block-scaled MXFP8 product on the tensor cores
  (tcgen05) that reads the cast's bytes as stored: the consumer check of the
  blocked scale layouts and the K-group slabs.

With MXQ_CHECKED=1 in the environment the binding loads libmxq_checked.so,
the same kernels with every computed global access tested against its buffer.
"""
from __future__ import annotations

import ctypes
import os
from pathlib import Path
from typing import NamedTuple, Optional

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libmxq.so"
CHECKED_LIB_PATH = _PKG / "libmxq_checked.so"

# status codes and constants of mxq.h
OK = 0
EBADSHAPE = -1
EBADDTYPE = -2
EBADOFFS = -3
EALIGN = -4
EOVERLAP = -5
ECUDA = -6
ENULL = -7
ESCRATCH = -8
F32 = 0
BF16 = 1
MAX_GROUPS = 1024
FMT_MX9 = 9
FMT_MX6 = 6
RECORD_BYTES = {FMT_MX9: 18, FMT_MX6: 12}
DEV_BADOFFS = 0x1
DEV_TIMEOUT = 0x2
DEV_OOB = 0x4  # checked library only: an out-of-buffer access was skipped

_lib: Optional[ctypes.CDLL] = None


class MxqError(RuntimeError):
    """A call into libmxq.so returned a non-zero status."""

    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (status {code})")


def lib() -> ctypes.CDLL:
    """Load libmxq.so (built by ``__graft_entry__.build()``); raise if it is missing.
    With MXQ_CHECKED=1 in the environment, load the bounds-checked twin
    libmxq_checked.so instead (same results; out-of-buffer accesses skipped and
    reported as MXQ_DEV_OOB in the device status word)."""
    global _lib
    if _lib is None:
        path = CHECKED_LIB_PATH if os.environ.get("MXQ_CHECKED") == "1" else LIB_PATH
        if not path.exists():
            raise ImportError(
                f"{path.name} is not built; run `python -c 'import __graft_entry__ as g; "
                f"g.build()'` (there is no CPU fallback)")
        L = ctypes.CDLL(str(path))
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        L.mxq_quantize_2d_dual.restype = ctypes.c_int
        L.mxq_quantize_2d_dual.argtypes = [vp, i64, i64, vp, i32, vp, vp, vp, vp, vp]
        L.mxq_quantize_2d_dual_rows.restype = ctypes.c_int
        L.mxq_quantize_2d_dual_rows.argtypes = [vp, i64, i64, i64, i64, vp, i32, vp, vp, vp, vp, vp]
        L.mx9_pack.restype = ctypes.c_int
        L.mx9_pack.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp, vp, vp]
        L.mx9_unpack.restype = ctypes.c_int
        L.mx9_unpack.argtypes = [vp, vp, vp, vp, ctypes.c_int, i64, i64, vp]
        L.mxq_quantize_1x32.restype = ctypes.c_int
        L.mxq_quantize_1x32.argtypes = [vp, i64, i64, vp, vp, vp]
        L.mxq_quantize_32x1.restype = ctypes.c_int
        L.mxq_quantize_32x1.argtypes = [vp, i64, i64, vp, vp, vp]
        L.mxq_swizzle_kgroups.restype = ctypes.c_int
        L.mxq_swizzle_kgroups.argtypes = [vp, i64, i64, vp, i32, vp, vp]
        L.mxq_quantize_2d_dual_3pass.restype = ctypes.c_int
        L.mxq_quantize_2d_dual_3pass.argtypes = [vp, i64, i64, vp, i32, vp, vp, vp, vp, vp, i64, vp]
        L.mx_pack_packed.restype = ctypes.c_int
        L.mx_pack_packed.argtypes = [vp, ctypes.c_int, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                     vp, vp]
        L.mx_unpack_packed.restype = ctypes.c_int
        L.mx_unpack_packed.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i64, i64, i64,
                                       ctypes.c_int, vp]
        L.mxq_mxfp8_scaled_mm.restype = ctypes.c_int
        L.mxq_mxfp8_scaled_mm.argtypes = [vp, i64, vp, vp, i64, vp, vp, i64, i64, i64, vp]
        L.mxq_last_device_status.restype = ctypes.c_int
        L.mxq_last_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        L.mxq_selftest_wait_timeout.restype = ctypes.c_int
        L.mxq_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.mxq_debug_bounds.restype = ctypes.c_int
        L.mxq_debug_bounds.argtypes = []
        L.mxq_selftest_bounds.restype = ctypes.c_int
        L.mxq_selftest_bounds.argtypes = [vp]
        L.mxq_device_status.restype = ctypes.c_int
        L.mxq_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        L.mxq_status_string.restype = ctypes.c_char_p
        L.mxq_status_string.argtypes = [ctypes.c_int]
        L.mxq_version.restype = ctypes.c_int
        L.mxq_version.argtypes = []
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().mxq_status_string(int(code)).decode()


def version() -> tuple[int, int]:
    v = lib().mxq_version()
    return v >> 16, v & 0xFFFF


def device_status(clear: bool = True) -> int:
    """Sticky MXQ_DEV_* bits of the current device (synchronizes the device)."""
    out = ctypes.c_uint32(0)
    rc = lib().mxq_device_status(ctypes.byref(out), int(bool(clear)))
    if rc != OK:
        raise MxqError(rc, "mxq_device_status")
    return int(out.value)


def selftest_wait_timeout(limit_ns: int = 50_000_000, stream=None) -> None:
    """Launch the bounded-wait self-test (see mxq.h); afterwards device_status()
    reports DEV_TIMEOUT."""
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    rc = lib().mxq_selftest_wait_timeout(int(limit_ns), ctypes.c_void_p(s.cuda_stream))
    if rc != OK:
        raise MxqError(rc, "mxq_selftest_wait_timeout")


def debug_bounds() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().mxq_debug_bounds())


def selftest_bounds(stream=None) -> None:
    """Launch the bounds-check self-test (see mxq.h); afterwards device_status()
    reports DEV_OOB in the checked library and nothing in the release one."""
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    rc = lib().mxq_selftest_bounds(ctypes.c_void_p(s.cuda_stream))
    if rc != OK:
        raise MxqError(rc, "mxq_selftest_bounds")


# ---------------------------------------------------------------------------
# torch-facing wrappers (marshalling only)
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _check_cuda(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(device, stream):
    torch = _torch()
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class DualOutputs(NamedTuple):
    q_row: "object"  # uint8 [M, N]    E4M3 bytes, 1x32 blocks along N
    s_row: "object"  # uint8 [M*N/32]  E8M0, blocked [M, N/32]
    q_col: "object"  # uint8 [N, M]    E4M3 bytes, 32x1 blocks along M, transposed
    s_col: "object"  # uint8 [N*M/32]  E8M0, per-group blocked slabs, zero tail


def quantize_2d_dual(x, offs=None, *, out: Optional[DualOutputs] = None, stream=None) -> DualOutputs:
    """Dual-axis MXFP8 cast of a bf16 CUDA tensor [M, N] (M, N multiples of 128).

    ``offs``: optional int32 CUDA tensor of cumulative group ends (multiples of
    128, non-decreasing, offs[-1] <= M); None means one dense group.
    Returns uint8 tensors; view them as torch.float8_e4m3fn / float8_e8m0fnu as
    needed.  An invalid ``offs`` is detected on the device: nothing is written
    and :func:`device_status` reports DEV_BADOFFS.
    """
    torch = _torch()
    _check_cuda(x, "x")
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    M, N = x.shape
    G = 0
    if offs is not None:
        _check_cuda(offs, "offs")
        if offs.dtype != torch.int32 or offs.dim() != 1:
            raise ValueError("offs must be a 1-D int32 tensor")
        if offs.device != x.device:
            raise ValueError("offs must be on x's device")
        G = offs.numel()
    if out is None:
        kw = dict(dtype=torch.uint8, device=x.device)
        out = DualOutputs(torch.empty((M, N), **kw), torch.empty((M * N // 32,), **kw),
                          torch.empty((N, M), **kw), torch.empty((N * M // 32,), **kw))
    for name, t, n in zip(DualOutputs._fields, out, (M * N, M * N // 32, M * N, M * N // 32)):
        _check_cuda(t, name)
        if t.dtype != torch.uint8 or t.numel() != n or t.device != x.device:
            raise ValueError(f"{name} must be a uint8 tensor of {n} elements on x's device")
    with torch.cuda.device(x.device):
        rc = lib().mxq_quantize_2d_dual(
            ctypes.c_void_p(x.data_ptr()), M, N,
            ctypes.c_void_p(offs.data_ptr() if offs is not None else 0), G,
            *(ctypes.c_void_p(t.data_ptr()) for t in out), _stream_handle(x.device, stream))
    if rc != OK:
        raise MxqError(rc, "mxq_quantize_2d_dual")
    return out


def quantize_2d_dual_rows(x, row0: int, M: int, s_col, offs=None, *, out=None, stream=None):
    """The dual-axis cast of rows [row0, row0 + x.shape[0]) of a full [M, N]
    tensor (a data-parallel band along M).  ``s_col`` is the FULL colwise
    scale buffer (uint8, N*M/32): this call writes the band's atoms only.
    ``offs`` are the full tensor's group ends.  Returns the band's q_row,
    s_row and q_col (q_col as [N, rows]) and s_col."""
    torch = _torch()
    _check_cuda(x, "x")
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    rows, N = x.shape
    G = 0
    if offs is not None:
        _check_cuda(offs, "offs")
        if offs.dtype != torch.int32 or offs.dim() != 1 or offs.device != x.device:
            raise ValueError("offs must be a 1-D int32 tensor on x's device")
        G = offs.numel()
    _check_cuda(s_col, "s_col")
    if s_col.dtype != torch.uint8 or s_col.numel() != N * M // 32 or s_col.device != x.device:
        raise ValueError("s_col must be the full uint8 colwise scale buffer (N*M/32) on x's device")
    if out is None:
        kw = dict(dtype=torch.uint8, device=x.device)
        out = (torch.empty((rows, N), **kw), torch.empty((rows * N // 32,), **kw),
               torch.empty((N, rows), **kw))
    q_row, s_row, q_col = out
    for name, t, n in (("q_row", q_row, rows * N), ("s_row", s_row, rows * N // 32),
                       ("q_col", q_col, rows * N)):
        _check_cuda(t, name)
        if t.dtype != torch.uint8 or t.numel() != n or t.device != x.device:
            raise ValueError(f"{name} must be a uint8 tensor of {n} elements on x's device")
    with torch.cuda.device(x.device):
        rc = lib().mxq_quantize_2d_dual_rows(
            ctypes.c_void_p(x.data_ptr()), rows, N, row0, M,
            ctypes.c_void_p(offs.data_ptr() if offs is not None else 0), G,
            ctypes.c_void_p(q_row.data_ptr()), ctypes.c_void_p(s_row.data_ptr()),
            ctypes.c_void_p(q_col.data_ptr()), ctypes.c_void_p(s_col.data_ptr()),
            _stream_handle(x.device, stream))
    if rc != OK:
        raise MxqError(rc, "mxq_quantize_2d_dual_rows")
    return DualOutputs(q_row, s_row, q_col, s_col)


def _check_x_offs(x, offs):
    torch = _torch()
    _check_cuda(x, "x")
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    G = 0
    if offs is not None:
        _check_cuda(offs, "offs")
        if offs.dtype != torch.int32 or offs.dim() != 1 or offs.device != x.device:
            raise ValueError("offs must be a 1-D int32 tensor on x's device")
        G = offs.numel()
    return G


def _u8(t, n, name, device):
    torch = _torch()
    _check_cuda(t, name)
    if t.dtype != torch.uint8 or t.numel() != n or t.device != device:
        raise ValueError(f"{name} must be a uint8 tensor of {n} elements on x's device")


def quantize_1x32(x, *, out=None, stream=None):
    """Rowwise-only cast: (q_row [M, N], s_row [M*N/32] blocked), as quantize_2d_dual."""
    torch = _torch()
    _check_x_offs(x, None)
    M, N = x.shape
    kw = dict(dtype=torch.uint8, device=x.device)
    q_row, s_row = out if out is not None else (torch.empty((M, N), **kw),
                                                torch.empty((M * N // 32,), **kw))
    _u8(q_row, M * N, "q_row", x.device)
    _u8(s_row, M * N // 32, "s_row", x.device)
    with torch.cuda.device(x.device):
        rc = lib().mxq_quantize_1x32(ctypes.c_void_p(x.data_ptr()), M, N,
                                     ctypes.c_void_p(q_row.data_ptr()),
                                     ctypes.c_void_p(s_row.data_ptr()),
                                     _stream_handle(x.device, stream))
    if rc != OK:
        raise MxqError(rc, "mxq_quantize_1x32")
    return q_row, s_row


def quantize_32x1(x, *, out=None, stream=None):
    """Colwise-only cast with the separate 32x1 cast's NaN rule: (q_col [N, M],
    s_rm [N, M/32] row-major scales)."""
    torch = _torch()
    _check_x_offs(x, None)
    M, N = x.shape
    kw = dict(dtype=torch.uint8, device=x.device)
    q_col, s_rm = out if out is not None else (torch.empty((N, M), **kw),
                                               torch.empty((N, M // 32), **kw))
    _u8(q_col, M * N, "q_col", x.device)
    _u8(s_rm, M * N // 32, "s_rm", x.device)
    with torch.cuda.device(x.device):
        rc = lib().mxq_quantize_32x1(ctypes.c_void_p(x.data_ptr()), M, N,
                                     ctypes.c_void_p(q_col.data_ptr()),
                                     ctypes.c_void_p(s_rm.data_ptr()),
                                     _stream_handle(x.device, stream))
    if rc != OK:
        raise MxqError(rc, "mxq_quantize_32x1")
    return q_col, s_rm


def swizzle_kgroups(s_rm, offs=None, *, out=None, stream=None):
    """Row-major colwise scales [N, M/32] -> the fused cast's grouped blocked s_col."""
    torch = _torch()
    _check_cuda(s_rm, "s_rm")
    if s_rm.dtype != torch.uint8 or s_rm.dim() != 2:
        raise ValueError("s_rm must be a 2-D uint8 tensor [N, M/32]")
    N, C = s_rm.shape
    M = 32 * C
    G = 0
    if offs is not None:
        _check_cuda(offs, "offs")
        if offs.dtype != torch.int32 or offs.dim() != 1 or offs.device != s_rm.device:
            raise ValueError("offs must be a 1-D int32 tensor on s_rm's device")
        G = offs.numel()
    if out is None:
        out = torch.empty((N * M // 32,), dtype=torch.uint8, device=s_rm.device)
    _u8(out, N * M // 32, "s_col", s_rm.device)
    with torch.cuda.device(s_rm.device):
        rc = lib().mxq_swizzle_kgroups(ctypes.c_void_p(s_rm.data_ptr()), N, M,
                                       ctypes.c_void_p(offs.data_ptr() if offs is not None else 0),
                                       G, ctypes.c_void_p(out.data_ptr()),
                                       _stream_handle(s_rm.device, stream))
    if rc != OK:
        raise MxqError(rc, "mxq_swizzle_kgroups")
    return out


def quantize_2d_dual_3pass(x, offs=None, *, workspace=None, out=None, stream=None) -> DualOutputs:
    """The three-pass composition (1x32, 32x1, swizzle) with a caller workspace of
    >= M*N/32 bytes (allocated here when not given)."""
    torch = _torch()
    G = _check_x_offs(x, offs)
    M, N = x.shape
    kw = dict(dtype=torch.uint8, device=x.device)
    if out is None:
        out = DualOutputs(torch.empty((M, N), **kw), torch.empty((M * N // 32,), **kw),
                          torch.empty((N, M), **kw), torch.empty((N * M // 32,), **kw))
    for name, t, n in zip(DualOutputs._fields, out, (M * N, M * N // 32, M * N, M * N // 32)):
        _u8(t, n, name, x.device)
    if workspace is None:
        workspace = torch.empty((max(M * N // 32, 16),), **kw)
    _check_cuda(workspace, "workspace")
    with torch.cuda.device(x.device):
        rc = lib().mxq_quantize_2d_dual_3pass(
            ctypes.c_void_p(x.data_ptr()), M, N,
            ctypes.c_void_p(offs.data_ptr() if offs is not None else 0), G,
            *(ctypes.c_void_p(t.data_ptr()) for t in out),
            ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(),
            _stream_handle(x.device, stream))
    if rc != OK:
        raise MxqError(rc, "mxq_quantize_2d_dual_3pass")
    return out


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise ValueError("dtype must be float32 or bfloat16")


def mx9_pack(x, *, out=None, stream=None):
    """MX9 pack of a fp32/bf16 CUDA tensor [rows, cols], cols % 16 == 0.

    Returns (q int8 [n_blocks, 16], max_exp uint8 [n_blocks], prime uint8 [n_blocks, 1]).
    """
    torch = _torch()
    _check_cuda(x, "x")
    dt = _dtype_code(x)
    if x.dim() != 2:
        raise ValueError("x must be 2-D")
    rows, cols = x.shape
    nb = rows * cols // 16
    if out is None:
        out = (torch.empty((nb, 16), dtype=torch.int8, device=x.device),
               torch.empty((nb,), dtype=torch.uint8, device=x.device),
               torch.empty((nb, 1), dtype=torch.uint8, device=x.device))
    q, e, p = out
    for name, t, dtype, n in (("q", q, torch.int8, nb * 16), ("max_exp", e, torch.uint8, nb),
                              ("prime", p, torch.uint8, nb)):
        _check_cuda(t, name)
        if t.dtype != dtype or t.numel() != n or t.device != x.device:
            raise ValueError(f"{name}: expected {dtype} with {n} elements on x's device")
    with torch.cuda.device(x.device):
        rc = lib().mx9_pack(ctypes.c_void_p(x.data_ptr()), dt, rows, cols,
                            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(e.data_ptr()),
                            ctypes.c_void_p(p.data_ptr()), _stream_handle(x.device, stream))
    if rc != OK:
        raise MxqError(rc, "mx9_pack")
    return q, e, p


def mx9_unpack(q, max_exp, prime, out_dtype, shape, *, out=None, stream=None):
    """Rebuild a [rows, cols] fp32/bf16 CUDA tensor from the MX9 parts (shape is passed back)."""
    torch = _torch()
    rows, cols = shape
    nb = rows * cols // 16
    for name, t, dtype, n in (("q", q, torch.int8, nb * 16), ("max_exp", max_exp, torch.uint8, nb),
                              ("prime", prime, torch.uint8, nb)):
        _check_cuda(t, name)
        if t.dtype != dtype or t.numel() != n or t.device != q.device:
            raise ValueError(f"{name}: expected {dtype} with {n} elements on q's device")
    if out is None:
        out = torch.empty((rows, cols), dtype=out_dtype, device=q.device)
    _check_cuda(out, "out")
    if out.dtype != out_dtype or out.numel() != rows * cols or out.device != q.device:
        raise ValueError("out must match out_dtype, shape and q's device")
    dt = _dtype_code(out)
    with torch.cuda.device(q.device):
        rc = lib().mx9_unpack(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(max_exp.data_ptr()),
                              ctypes.c_void_p(prime.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                              dt, rows, cols, _stream_handle(q.device, stream))
    if rc != OK:
        raise MxqError(rc, "mx9_unpack")
    return out


# ---------------------------------------------------------------------------
# MX9 / MX6 in one packed tensor, any axis, strided views, padded blocks
# ---------------------------------------------------------------------------

def _view_2d(t, name):
    """(rows, cols, ld) of a 2-D CUDA tensor whose rows may be strided."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if t.dim() != 2 or t.stride(1) != 1 or (t.shape[0] > 1 and t.stride(0) < t.shape[1]):
        raise ValueError(f"{name} must be 2-D with unit column stride")
    rows, cols = t.shape
    return rows, cols, (t.stride(0) if rows > 1 else cols)


def mx_blocks(rows: int, cols: int, axis: int) -> int:
    lines, length = (rows, cols) if axis == 1 else (cols, rows)
    return lines * ((length + 15) // 16)


def mx_pack_packed(x, fmt: int = FMT_MX9, axis: int = 1, *, out=None, stream=None):
    """Pack a fp32/bf16 CUDA tensor (strided rows allowed) into uint8 records
    [n_blocks, 18 (MX9) or 12 (MX6)], blocks of 16 along `axis`."""
    torch = _torch()
    if fmt not in RECORD_BYTES:
        raise ValueError(f"unknown MX format {fmt} (FMT_MX9 or FMT_MX6)")
    dt = _dtype_code(x)
    rows, cols, ld = _view_2d(x, "x")
    nb = mx_blocks(rows, cols, axis)
    if out is None:
        out = torch.empty((nb, RECORD_BYTES[fmt]), dtype=torch.uint8, device=x.device)
    _check_cuda(out, "out")
    if out.dtype != torch.uint8 or out.numel() != nb * RECORD_BYTES[fmt] or out.device != x.device:
        raise ValueError("out must be uint8 [n_blocks, record bytes] on x's device")
    with torch.cuda.device(x.device):
        rc = lib().mx_pack_packed(ctypes.c_void_p(x.data_ptr()), dt, rows, cols, ld, axis, fmt,
                                  ctypes.c_void_p(out.data_ptr()), _stream_handle(x.device, stream))
    if rc != OK:
        raise MxqError(rc, "mx_pack_packed")
    return out


def mx_unpack_packed(packed, fmt: int, out, axis: int = 1, *, stream=None):
    """Rebuild into `out` (a fp32/bf16 CUDA tensor, strided rows allowed) from
    records produced by mx_pack_packed with the same shape and axis."""
    torch = _torch()
    if fmt not in RECORD_BYTES:
        raise ValueError(f"unknown MX format {fmt} (FMT_MX9 or FMT_MX6)")
    dt = _dtype_code(out)
    rows, cols, ld = _view_2d(out, "out")
    _check_cuda(packed, "packed")
    nb = mx_blocks(rows, cols, axis)
    if packed.dtype != torch.uint8 or packed.numel() != nb * RECORD_BYTES[fmt]:
        raise ValueError("packed must be uint8 [n_blocks, record bytes] for this shape")
    with torch.cuda.device(out.device):
        rc = lib().mx_unpack_packed(ctypes.c_void_p(packed.data_ptr()), fmt,
                                    ctypes.c_void_p(out.data_ptr()), dt, rows, cols, ld, axis,
                                    _stream_handle(out.device, stream))
    if rc != OK:
        raise MxqError(rc, "mx_unpack_packed")
    return out


# ---------------------------------------------------------------------------
# consumer check of the layouts: a block-scaled MXFP8 product on the tensor cores
# ---------------------------------------------------------------------------

def mxfp8_scaled_mm(a, sa, b, sb, *, out=None, stream=None):
    """fp32 [Ma, Nb] = (a scaled by sa) @ (b scaled by sb)^T on tcgen05.

    ``a``: uint8 E4M3 [Ma, K] CUDA tensor whose rows may be strided (unit column
    stride, row stride a multiple of 16), e.g. ``q_row`` or the K-group columns
    ``q_col[:, lo:hi]``; ``sa``: uint8 E8M0 [Ma*K/32] in the 128x4 blocked layout
    (``s_row``, or the group's slab of ``s_col``).  Likewise ``b``/``sb``.
    Ma, Nb, K multiples of 128."""
    torch = _torch()
    ma, k, lda = _view_2d(a, "a")
    nb, kb, ldb = _view_2d(b, "b")
    if k != kb:
        raise ValueError(f"a and b disagree on K: {k} vs {kb}")
    for t, name, n in ((sa, "sa", ma * k // 32), (sb, "sb", nb * k // 32)):
        _check_cuda(t, name)
        if t.dtype != torch.uint8 or t.numel() != n:
            raise ValueError(f"{name} must be uint8 with {n} bytes")
    if a.dtype != torch.uint8 or b.dtype != torch.uint8:
        raise ValueError("a and b must be uint8 E4M3 bytes")
    if out is None:
        out = torch.empty((ma, nb), dtype=torch.float32, device=a.device)
    _check_cuda(out, "out")
    if out.dtype != torch.float32 or tuple(out.shape) != (ma, nb):
        raise ValueError(f"out must be float32 [{ma}, {nb}]")
    vp = ctypes.c_void_p
    with torch.cuda.device(a.device):
        rc = lib().mxq_mxfp8_scaled_mm(vp(a.data_ptr()), lda, vp(sa.data_ptr()), vp(b.data_ptr()), ldb,
                                       vp(sb.data_ptr()), vp(out.data_ptr()), ma, nb, k,
                                       _stream_handle(a.device, stream))
    if rc != OK:
        raise MxqError(rc, "mxq_mxfp8_scaled_mm")
    return out

