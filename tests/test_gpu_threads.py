"""Calls from several host threads at once, in a fresh process so that each
kernel's first-call setup (shared-memory attribute, occupancy and per-device
caches) is reached by the threads concurrently: every result still equals the
oracle byte for byte.  ctypes releases the interpreter lock during a foreign
call, so the threads really are inside the library together."""
import os
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest

from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


CHILD = textwrap.dedent("""
    import sys, threading
    import numpy as np, torch
    import mx_block_quantization_gb300 as mxq
    import oracle
    from mx_block_quantization_gb300 import workloads as W

    def work(t, errors):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            xa, oa = W.moe_grouped(M=2048, N=1024, experts=4, routed_units=12, seed=60 + t)
            xm = W.mx9_outliers(512, 1024, seed=70 + t)
            xc = W.mx9_outliers(256, 384, seed=80 + t, zero_blocks=0, tiny_blocks=0)
            with torch.cuda.stream(s):
                da = torch.from_numpy(xa.view(np.int16)).view(torch.bfloat16).cuda()
                offs = torch.from_numpy(oa).cuda()
                dm = torch.from_numpy(xm).cuda()
                dc = torch.from_numpy(xc).cuda()
                for rep in range(3):
                    out = mxq.quantize_2d_dual(da, offs, stream=s)
                    q, e, p = mxq.mx9_pack(dm, stream=s)
                    y = mxq.mx9_unpack(q, e, p, torch.float32, xm.shape, stream=s)
                    rec = mxq.mx_pack_packed(dc, mxq.FMT_MX9, 0, stream=s)   # column tiles
                    yc = torch.empty_like(dc)
                    mxq.mx_unpack_packed(rec, mxq.FMT_MX9, yc, 0, stream=s)
            s.synchronize()
            want = oracle.mxfp8_dual(xa, oa)
            for k in out._fields:
                assert np.array_equal(getattr(out, k).cpu().numpy().reshape(-1), want[k]), (t, k)
            rq, re, rp = oracle.mx9_pack(xm)
            assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(e.cpu().numpy(), re), t
            ry = oracle.mx9_unpack(rq, re, rp, "f32", *xm.shape)
            assert np.array_equal(y.cpu().numpy().view(np.uint32), ry.view(np.uint32)), t
            wrec = oracle.mx_pack(xc, mxq.FMT_MX9, axis=0)
            assert np.array_equal(rec.cpu().numpy(), wrec), (t, "records")
            wy = oracle.mx_unpack(wrec, mxq.FMT_MX9, *xc.shape, "f32", axis=0)
            assert np.array_equal(yc.cpu().numpy().view(np.uint32), wy.view(np.uint32)), (t, "cols")
        except BaseException as ex:  # reported by the main thread
            errors.append(repr(ex))

    errors = []
    threads = [threading.Thread(target=work, args=(t, errors)) for t in range(4)]
    for th in threads: th.start()
    for th in threads: th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert mxq.device_status(clear=True) == 0
    print("ok")
""")


def test_four_threads_from_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=dict(os.environ),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, (r.stdout + r.stderr)[-3000:]
