"""Helpers for the GPU parity tests: device transfer, 0xAB-prefilled outputs and
byte comparisons that name the first mismatch."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import mx_block_quantization_gb300 as mxq

FILL = 0xAB


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from mx_block_quantization_gb300.build import build_library
    build_library(checked=os.environ.get("MXQ_CHECKED") == "1")  # the library lib() loads
    mxq.device_status(clear=True)


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dual_outputs(M: int, N: int, fill: int = FILL) -> mxq.DualOutputs:
    kw = dict(dtype=torch.uint8, device="cuda")
    return mxq.DualOutputs(torch.full((M, N), fill, **kw), torch.full((M * N // 32,), fill, **kw),
                           torch.full((N, M), fill, **kw), torch.full((M * N // 32,), fill, **kw))


def run_dual(bits: np.ndarray, offs: np.ndarray | None, fill: int = FILL, stream=None):
    M, N = bits.shape
    x = to_dev_bf16(bits)
    o = None if offs is None else torch.from_numpy(np.asarray(offs, np.int32)).cuda()
    out = dual_outputs(M, N, fill)
    mxq.quantize_2d_dual(x, o, out=out, stream=stream)
    torch.cuda.synchronize()
    return {k: getattr(out, k).cpu().numpy().reshape(-1) for k in out._fields}


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got).reshape(-1)
    want = np.asarray(want).reshape(-1)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    bad = np.flatnonzero(got != want)
    if bad.size:
        i = int(bad[0])
        raise AssertionError(f"{what}: {bad.size} bytes differ; first at flat index {i}: "
                             f"got {int(got[i]):#x} want {int(want[i]):#x}")


def assert_dual_equal(got: dict, want: dict, tag: str = ""):
    for k in ("q_row", "s_row", "q_col", "s_col"):
        assert_bytes_equal(got[k], want[k], f"{tag}{k}")
