"""Seeded fuzz of the C ABI's host-side argument checks, without a GPU.

Sizes are drawn from edge values (0, 1, the method's multiples and their
neighbours, 2^31 - 1, 2^31, 2^40, 2^62, INT64_MAX and negatives), pointers are
well separated 16-byte aligned fake addresses (never dereferenced on the host).
For every call the result must be what the shape rules alone decide:
MXQ_EBADSHAPE for a shape the rules reject, MXQ_OK for an empty problem (no work,
no CUDA call), and otherwise a call that gets past the checks and stops at the
first CUDA call (MXQ_ECUDA here) or, for sizes too large to fit between the fake
buffers, MXQ_EOVERLAP.  The calls run in a child process, so a crash fails the
test instead of ending the run; nothing here runs where a GPU is visible, since
fake pointers must never reach a kernel launch.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, ROOT)
import mx_block_quantization_gb300 as mxq
L = mxq.lib()
vp = ctypes.c_void_p
# not wrapped by the binding: declared here so 64-bit sizes pass unchanged
L.mxq_quantize_2d_dual_3pass_noalloc.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp,
                                                 ctypes.c_int32, vp, vp, vp, vp, vp]
L.mxq_quantize_2d_dual_3pass_noalloc.restype = ctypes.c_int
I64_MAX = (1 << 63) - 1
EDGE = [0, 1, 15, 16, 17, 31, 32, 127, 128, 129, 256, 4096, 8192 + 128, (1 << 31) - 1, 1 << 31,
        (1 << 31) + 128, 1 << 40, 1 << 62, I64_MAX - 127, I64_MAX, -1, -128, -(1 << 62)]
g = np.random.Generator(np.random.PCG64(20261202))
BASE = [(k + 1) << 56 for k in range(8)]  # buffers 2^56 bytes apart
def pick():
    return int(EDGE[g.integers(len(EDGE))]) if g.random() < 0.8 else int(g.integers(-4, 1 << 20)) * 16
bad = []
seen = {}
def expect(name, got, want, args):
    seen[got] = seen.get(got, 0) + 1
    if got not in want:
        bad.append((name, args, got, sorted(want)))
for _ in range(N_CASES):
    # dual-axis cast, dense
    M, N = pick(), pick()
    rc = L.mxq_quantize_2d_dual(vp(BASE[0]), M, N, None, 0, vp(BASE[1]), vp(BASE[2]), vp(BASE[3]),
                                vp(BASE[4]), None)
    ok_shape = M >= 0 and N >= 0 and M % 128 == 0 and N % 128 == 0 and M <= (1 << 31) - 1 and N <= (1 << 31) - 1
    if not ok_shape:
        want = {mxq.EBADSHAPE}
    elif M * N == 0:
        want = {mxq.OK}
    else:
        want = {mxq.ECUDA, mxq.EOVERLAP}
    expect("dual", rc, want, (M, N))
    dual_shape = ok_shape
    # the single-axis casts and the three passes take the same shapes
    rc = L.mxq_quantize_1x32(vp(BASE[0]), M, N, vp(BASE[1]), vp(BASE[2]), None)
    expect("1x32", rc, want, (M, N))
    rc = L.mxq_quantize_32x1(vp(BASE[0]), M, N, vp(BASE[3]), vp(BASE[4]), None)
    expect("32x1", rc, want, (M, N))
    rc = L.mxq_swizzle_kgroups(vp(BASE[4]), N, M, None, 0, vp(BASE[5]), None)
    expect("swizzle", rc, want, (M, N))
    ws = pick()
    rc = L.mxq_quantize_2d_dual_3pass(vp(BASE[0]), M, N, None, 0, vp(BASE[1]), vp(BASE[2]),
                                      vp(BASE[3]), vp(BASE[4]), vp(BASE[6]), ws, None)
    want3 = want if not dual_shape or M * N == 0 else \
        ({mxq.EBADSHAPE} if ws < 0 or ws < M * N // 32 else want)
    expect("3pass", rc, want3, (M, N, ws))
    rc = L.mxq_quantize_2d_dual_3pass_noalloc(vp(BASE[0]), M, N, None, 0, vp(BASE[1]), vp(BASE[2]),
                                              vp(BASE[3]), vp(BASE[4]), None)
    wantn = want if not dual_shape or M * N == 0 else \
        ({mxq.ESCRATCH} if M * N // 32 > (16 << 20) else want)
    expect("3pass_noalloc", rc, wantn, (M, N))
    # one band [row0, row0 + rows) of an M-row matrix
    rows, row0 = pick(), pick()
    rc = L.mxq_quantize_2d_dual_rows(vp(BASE[0]), rows, N, row0, M, None, 0, vp(BASE[1]),
                                     vp(BASE[2]), vp(BASE[3]), vp(BASE[4]), None)
    shape_ok = lambda a: a >= 0 and a % 128 == 0 and a <= (1 << 31) - 1
    band_ok = shape_ok(rows) and dual_shape and row0 >= 0 and row0 % 128 == 0 and row0 + rows <= M
    wantr = {mxq.EBADSHAPE} if not band_ok else {mxq.OK} if rows * N == 0 else {mxq.ECUDA, mxq.EOVERLAP}
    expect("dual_rows", rc, wantr, (rows, N, row0, M))
    # split MX9 pack and unpack
    rows, cols, dt = pick(), pick(), int(g.integers(0, 2))
    rc = L.mx9_pack(vp(BASE[0]), dt, rows, cols, vp(BASE[1]), vp(BASE[2]), vp(BASE[3]), None)
    ok_shape = rows >= 0 and cols >= 0 and cols % 16 == 0 and (cols == 0 or rows <= (I64_MAX // 8) // cols)
    want = {mxq.EBADSHAPE} if not ok_shape else {mxq.OK} if rows * cols == 0 else {mxq.ECUDA, mxq.EOVERLAP}
    expect("mx9_pack", rc, want, (rows, cols, dt))
    rc = L.mx9_unpack(vp(BASE[1]), vp(BASE[2]), vp(BASE[3]), vp(BASE[0]), dt, rows, cols, None)
    expect("mx9_unpack", rc, want, (rows, cols, dt))
    # packed MX9 / MX6, either axis, pitch >= cols
    ld = cols + (int(g.integers(0, 3)) * 16 if g.random() < 0.5 else pick())
    ld = (ld + (1 << 63)) % (1 << 64) - (1 << 63)  # the int64 the call receives
    axis, fmt = int(g.integers(0, 2)), (9, 6)[int(g.integers(0, 2))]
    rc = L.mx_pack_packed(vp(BASE[0]), dt, rows, cols, ld, axis, fmt, vp(BASE[1]), None)
    ok_shape = rows >= 0 and cols >= 0 and ld >= cols and not (rows > 0 and ld > 0 and rows > (I64_MAX // 8) // ld)
    lines, length = (rows, cols) if axis == 1 else (cols, rows)
    empty = ok_shape and lines * ((length + 15) // 16) == 0
    want = {mxq.EBADSHAPE} if not ok_shape else {mxq.OK} if empty else {mxq.ECUDA, mxq.EOVERLAP}
    expect("mx_pack_packed", rc, want, (rows, cols, ld, axis, fmt, dt))
    rc = L.mx_unpack_packed(vp(BASE[1]), fmt, vp(BASE[0]), dt, rows, cols, ld, axis, None)
    expect("mx_unpack_packed", rc, want, (rows, cols, ld, axis, fmt, dt))
    # the tensor-core consumer check: Ma, Nb, K multiples of 128 up to 2^24, row pitches
    Ma, Nb, K = pick(), pick(), pick()
    lda = K + int(g.integers(0, 3)) * 16 if g.random() < 0.7 else pick()
    ldb = K if g.random() < 0.7 else pick()
    dims_ok = all(v >= 0 and v % 128 == 0 and v <= (1 << 24) for v in (Ma, Nb, K))
    rc = L.mxq_mxfp8_scaled_mm(vp(BASE[0]), lda, vp(BASE[1]), vp(BASE[2]), ldb, vp(BASE[3]),
                               vp(BASE[4]), Ma, Nb, K, None)
    if not dims_ok:
        want = {mxq.EBADSHAPE}
    elif Ma * Nb == 0:
        want = {mxq.OK}
    elif K == 0 or not all(l >= K and l % 16 == 0 and l <= (1 << 40) for l in (lda, ldb)):
        want = {mxq.EBADSHAPE}
    else:
        want = {mxq.ECUDA, mxq.EOVERLAP}
    expect("mxfp8_scaled_mm", rc, want, (Ma, Nb, K, lda, ldb))
# bands placed past int64 range by their start (row0 + rows would wrap)
for row0 in (I64_MAX - 127, I64_MAX - 255, (1 << 62) + 128, (1 << 31) * 128):
    for rows in (128, 256, 1 << 30):
        rc = L.mxq_quantize_2d_dual_rows(vp(BASE[0]), rows, 128, row0, 1 << 20, None, 0, vp(BASE[1]),
                                         vp(BASE[2]), vp(BASE[3]), vp(BASE[4]), None)
        expect("dual_rows far row0", rc, {mxq.EBADSHAPE}, (rows, row0))
# a buffer whose byte range would wrap past the top of the address space
TOP = (1 << 64) - 4096
for M, N in ((128, 128), (1024, 4096)):
    rc = L.mxq_quantize_2d_dual(vp(TOP), M, N, None, 0, vp(BASE[1]), vp(BASE[2]), vp(BASE[3]),
                                vp(BASE[4]), None)
    expect("dual wrapped x", rc, {mxq.EOVERLAP}, (M, N))
    rc = L.mx9_pack(vp(BASE[0]), 0, M, N, vp(TOP), vp(BASE[2]), vp(BASE[3]), None)
    expect("mx9_pack wrapped q", rc, {mxq.EOVERLAP}, (M, N))
    rc = L.mx_pack_packed(vp(TOP), 0, M, N, N, 1, 9, vp(BASE[1]), None)
    expect("mx_pack_packed wrapped x", rc, {mxq.EOVERLAP}, (M, N))
print("SEEN", seen.get(mxq.EBADSHAPE, 0), seen.get(mxq.OK, 0), seen.get(mxq.ECUDA, 0))
print("BAD", len(bad))
for b in bad[:20]:
    print(b)
'''


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers: host-only fuzz, never where a GPU is visible")
def test_host_checks_under_fuzz():
    import mx_block_quantization_gb300 as mxq
    if not mxq.LIB_PATH.exists():
        import __graft_entry__
        __graft_entry__.build()
    code = CHILD.replace("ROOT", repr(ROOT)).replace("N_CASES", "3000")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, f"child crashed or failed (rc {r.returncode}):\n{r.stderr[-3000:]}"
    assert "BAD 0" in r.stdout, r.stdout[-3000:]
    # every outcome occurs often: rejected shapes, empty problems, calls that reach CUDA
    seen = [int(v) for v in r.stdout.split("SEEN")[1].split()[:3]]
    assert min(seen) >= 200, seen
