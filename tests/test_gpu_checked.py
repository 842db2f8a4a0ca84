"""The bounds-checked build (libmxq_checked.so, MXQ_DEBUG_BOUNDS=1): a stand-in
for a memory checker where none can run.  Every computed global access of the
kernels outside the TMA tensor copies is tested against its buffer; one that
would leave it is skipped and reported as MXQ_DEV_OOB.  The whole GPU parity
suite runs again on that library in a child process: every module ends by
asserting a clean status word, so a single out-of-buffer access anywhere
fails it.  The checker itself is shown to report by a self-test that tests a
range past a dummy buffer without touching memory."""
import os
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest
import torch

import mx_block_quantization_gb300 as mxq
from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    assert mxq.device_status(clear=True) == 0


def _child(code: str, timeout: int = 600) -> subprocess.CompletedProcess:
    env = dict(os.environ, MXQ_CHECKED="1")
    return subprocess.run([sys.executable, "-c", textwrap.dedent(code)], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_release_library_has_no_checks():
    assert not mxq.debug_bounds()
    mxq.device_status(clear=True)
    mxq.selftest_bounds()
    torch.cuda.synchronize()
    assert mxq.device_status(clear=True) == 0


def test_checked_library_reports_a_range_past_its_buffer():
    r = _child("""
        from mx_block_quantization_gb300.build import build_library
        build_library(checked=True)
        import torch, mx_block_quantization_gb300 as mxq
        assert mxq.debug_bounds()
        mxq.device_status(clear=True)
        mxq.selftest_bounds()
        torch.cuda.synchronize()
        st = mxq.device_status(clear=True)
        assert st == mxq.DEV_OOB, st
        assert mxq.device_status(clear=True) == 0
        print("ok")
    """)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_gpu_suite_on_the_checked_library():
    files = sorted(str(p.relative_to(ROOT)) for p in (ROOT / "tests").glob("test_gpu_*.py")
                   if p.name != Path(__file__).name)
    r = _child(f"""
        import sys, pytest
        from mx_block_quantization_gb300.build import build_library
        build_library(checked=True)
        import mx_block_quantization_gb300 as mxq
        assert mxq.debug_bounds(), "the child must load the checked library"
        sys.exit(pytest.main({files!r} + ["-m", "gpu", "-q", "-x", "-p", "no:cacheprovider"]))
    """, timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
