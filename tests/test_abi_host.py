"""The C ABI library loads, exports every function declared in include/mxq.h, and
rejects bad arguments on the host (these paths make no CUDA call, so they run
without a GPU)."""
import ctypes
import os
import re

import pytest

import mx_block_quantization_gb300 as mxq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def L():
    if not mxq.LIB_PATH.exists():
        import __graft_entry__
        __graft_entry__.build()
    return mxq.lib()


def test_header_declares_the_entry_points():
    names = set(_declared_functions())
    assert {"mxq_quantize_2d_dual", "mx9_pack", "mx9_unpack", "mxq_device_status",
            "mxq_status_string", "mxq_version"} <= names


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_checked_twin_exports_the_same_and_says_so(L):
    """libmxq_checked.so (bounds checks compiled in) has the same entry points;
    mxq_debug_bounds tells the two apart without touching a GPU."""
    import ctypes
    if not mxq.CHECKED_LIB_PATH.exists():
        from mx_block_quantization_gb300.build import build_library
        build_library(checked=True)
    C = ctypes.CDLL(str(mxq.CHECKED_LIB_PATH))
    for name in _declared_functions():
        assert hasattr(C, name), name
    assert C.mxq_debug_bounds() == 1
    assert L.mxq_debug_bounds() == 0


def test_status_strings_and_version(L):
    for code in (mxq.OK, mxq.EBADSHAPE, mxq.EBADDTYPE, mxq.EBADOFFS, mxq.EALIGN, mxq.EOVERLAP,
                 mxq.ECUDA, mxq.ENULL):
        s = mxq.status_string(code)
        assert s and s != "unknown status"
    assert mxq.status_string(12345) == "unknown status"
    assert mxq.version() == (1, 0)


A = 1 << 20  # fake, 16-byte aligned "device addresses": never dereferenced


def _dual(L, x=A, M=128, N=128, offs=None, G=0, qr=None, sr=None, qc=None, sc=None):
    MN = M * N
    qr = A + 4 * MN if qr is None else qr
    qc = A + 8 * MN if qc is None else qc
    sr = A + 12 * MN if sr is None else sr
    sc = A + 14 * MN if sc is None else sc
    return L.mxq_quantize_2d_dual(ctypes.c_void_p(x), M, N, ctypes.c_void_p(offs), G,
                                  ctypes.c_void_p(qr), ctypes.c_void_p(sr), ctypes.c_void_p(qc),
                                  ctypes.c_void_p(sc), None)


def test_dual_rejections(L):
    assert _dual(L, M=100) == mxq.EBADSHAPE
    assert _dual(L, N=96) == mxq.EBADSHAPE
    assert _dual(L, M=-128) == mxq.EBADSHAPE
    assert _dual(L, M=1 << 31) == mxq.EBADSHAPE
    assert _dual(L, offs=None, G=1) == mxq.EBADOFFS          # NULL offs needs G == 0
    assert _dual(L, offs=A + (1 << 30), G=0) == mxq.EBADOFFS  # offs needs G >= 1
    assert _dual(L, offs=A + (1 << 30), G=mxq.MAX_GROUPS + 1) == mxq.EBADOFFS
    assert _dual(L, offs=A + (1 << 30) + 2, G=4) == mxq.EALIGN
    assert _dual(L, x=0) == mxq.ENULL
    assert _dual(L, sc=0) == mxq.ENULL
    assert _dual(L, x=A + 8) == mxq.EALIGN
    assert _dual(L, qc=A + 8 * 128 * 128 + 4) == mxq.EALIGN
    assert _dual(L, qr=A + 128 * 128) == mxq.EOVERLAP         # q_row inside x
    assert _dual(L, sr=A + 8 * 128 * 128 + 16) == mxq.EOVERLAP  # s_row inside q_col
    assert _dual(L, offs=A + 64, G=4) == mxq.EOVERLAP           # offs inside x
    # empty problems are no-ops that touch nothing (NULL pointers allowed)
    assert L.mxq_quantize_2d_dual(None, 0, 128, None, 0, None, None, None, None, None) == mxq.OK
    assert L.mxq_quantize_2d_dual(None, 128, 0, None, 0, None, None, None, None, None) == mxq.OK


def _pack(L, x=A, dtype=0, rows=4, cols=16, q=A + 4096, e=A + 8192, p=A + 12288):
    return L.mx9_pack(ctypes.c_void_p(x), dtype, rows, cols, ctypes.c_void_p(q),
                      ctypes.c_void_p(e), ctypes.c_void_p(p), None)


def _unpack(L, q=A, e=A + 4096, p=A + 8192, y=A + 12288, dtype=0, rows=4, cols=16):
    return L.mx9_unpack(ctypes.c_void_p(q), ctypes.c_void_p(e), ctypes.c_void_p(p),
                        ctypes.c_void_p(y), dtype, rows, cols, None)


def test_mx9_rejections(L):
    assert _pack(L, dtype=2) == mxq.EBADDTYPE
    assert _pack(L, cols=15) == mxq.EBADSHAPE
    assert _pack(L, rows=-1) == mxq.EBADSHAPE
    assert _pack(L, x=0) == mxq.ENULL
    assert _pack(L, x=A + 4) == mxq.EALIGN
    assert _pack(L, q=A + 16) == mxq.EOVERLAP  # q inside x (x spans 256 bytes)
    assert _pack(L, e=A + 4096 + 32) == mxq.EOVERLAP
    assert _pack(L, rows=0) == mxq.OK
    assert _unpack(L, dtype=7) == mxq.EBADDTYPE
    assert _unpack(L, cols=8) == mxq.EBADSHAPE
    assert _unpack(L, y=0) == mxq.ENULL
    assert _unpack(L, y=A + 12288 + 8) == mxq.EALIGN
    assert _unpack(L, y=A + 16) == mxq.EOVERLAP
    assert _unpack(L, cols=0) == mxq.OK


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros((128, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mxq.quantize_2d_dual(x)
    with pytest.raises(ValueError):
        mxq.mx9_pack(torch.zeros((4, 16)))


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_fails_loudly(L):
    """With no GPU the first CUDA call fails and the library reports it (no CPU fallback)."""
    assert _dual(L) == mxq.ECUDA
    assert _pack(L) == mxq.ECUDA


def test_composition_rejections(L):
    vp = ctypes.c_void_p
    M = N = 128
    MN = M * N
    ok = dict(x=A, qr=A + 4 * MN, sr=A + 6 * MN, qc=A + 8 * MN, sc=A + 10 * MN, ws=A + 12 * MN)

    def three(x=None, ws=None, wsb=MN // 32, M=M, N=N, offs=None, G=0):
        a = dict(ok)
        if x is not None:
            a["x"] = x
        if ws is not None:
            a["ws"] = ws
        return L.mxq_quantize_2d_dual_3pass(vp(a["x"]), M, N, vp(offs), G, vp(a["qr"]), vp(a["sr"]),
                                            vp(a["qc"]), vp(a["sc"]), vp(a["ws"]), wsb, None)
    assert three(M=100) == mxq.EBADSHAPE
    assert three(wsb=MN // 32 - 1) == mxq.EBADSHAPE
    assert three(ws=0) == mxq.ENULL
    assert three(ws=A + 12 * MN + 8) == mxq.EALIGN
    assert three(ws=A + 4 * MN + 16) == mxq.EOVERLAP     # workspace inside q_row
    assert three(offs=None, G=2) == mxq.EBADOFFS
    assert L.mxq_quantize_1x32(vp(A), 96, 128, vp(A + 4 * MN), vp(A + 6 * MN), None) == mxq.EBADSHAPE
    assert L.mxq_quantize_1x32(vp(A), M, N, vp(A + 16), vp(A + 6 * MN), None) == mxq.EOVERLAP
    assert L.mxq_quantize_32x1(vp(A), M, N, vp(0), vp(A + 6 * MN), None) == mxq.ENULL
    assert L.mxq_quantize_32x1(vp(A), M, N, vp(A + 4 * MN), vp(A + 4 * MN + 16), None) == mxq.EOVERLAP
    assert L.mxq_swizzle_kgroups(vp(A), N, M, vp(0), 1, vp(A + MN), None) == mxq.EBADOFFS
    assert L.mxq_swizzle_kgroups(vp(A), N, M, vp(0), 0, vp(A + 16), None) == mxq.EOVERLAP
    assert L.mxq_swizzle_kgroups(vp(A), 0, M, vp(0), 0, vp(0), None) == mxq.OK


def test_packed_variant_rejections(L):
    vp = ctypes.c_void_p

    def pack(x=A, dtype=0, rows=4, cols=32, ld=32, axis=1, fmt=9, out=A + 8192):
        return L.mx_pack_packed(vp(x), dtype, rows, cols, ld, axis, fmt, vp(out), None)
    assert pack(fmt=7) == mxq.EBADDTYPE
    assert pack(dtype=3) == mxq.EBADDTYPE
    assert pack(ld=16) == mxq.EBADSHAPE
    assert pack(axis=2) == mxq.EBADSHAPE
    assert pack(x=0) == mxq.ENULL
    assert pack(x=A + 2) == mxq.EALIGN          # fp32 elements need 4-byte alignment
    assert pack(out=A + 1) == mxq.EALIGN        # MX9 records need 2-byte alignment
    assert pack(out=A + 64) == mxq.EOVERLAP
    assert pack(rows=0) == mxq.OK
    assert L.mx_unpack_packed(vp(A), 6, vp(A + 64), 0, 4, 32, 32, 1, None) == mxq.EOVERLAP
    assert L.mx_unpack_packed(vp(A + 2), 6, vp(A + 4096), 0, 4, 32, 32, 1, None) == mxq.EALIGN


def test_dual_rows_rejections_before_any_cuda_call(L):
    """The band entry checks its band, pointers and overlaps on the host."""
    vp = ctypes.c_void_p
    f = L.mxq_quantize_2d_dual_rows
    N, M, rows = 128, 512, 128
    RN = rows * N
    x, qr, sr, qc, sc = A, A + 4 * RN, A + 8 * RN, A + 12 * RN, A + 16 * RN

    def call(rows=rows, row0=0, M=M, x=x, qr=qr, sr=sr, qc=qc, sc=sc, offs=None, G=0):
        return f(vp(x), rows, N, row0, M, vp(offs), G, vp(qr), vp(sr), vp(qc), vp(sc), None)

    assert call(row0=64) == mxq.EBADSHAPE           # band start not a multiple of 128
    assert call(row0=512) == mxq.EBADSHAPE          # band past the tensor
    assert call(rows=256, row0=384) == mxq.EBADSHAPE
    assert call(row0=(1 << 63) - 128) == mxq.EBADSHAPE  # row0 + rows would wrap int64
    assert call(M=500) == mxq.EBADSHAPE
    assert call(rows=0) == mxq.OK                    # empty band: nothing to do
    assert call(x=0) == mxq.ENULL
    assert call(qc=qc + 8) == mxq.EALIGN
    assert call(sc=x + 64) == mxq.EOVERLAP           # the full s_col overlapping x
    assert call(offs=A + 32 * RN, G=0) == mxq.EBADOFFS
    assert call(offs=None, G=3) == mxq.EBADOFFS
