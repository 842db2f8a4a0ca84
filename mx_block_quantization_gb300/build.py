"""Build libmxq.so (the sm_103a kernels and the C ABI) in-tree with nvcc.

Translation units compile in parallel; the result is cached under a stamp that
hashes the sources, the flags and the host machine, so a tree copied to another
machine (or architecture) rebuilds instead of loading a foreign binary.
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD_DIR = PKG / "_build"
LIB_PATH = PKG / "libmxq.so"
STAMP = BUILD_DIR / "libmxq.stamp"
# the checked build: every computed global access tested against its buffer
# (MXQ_DEBUG_BOUNDS=1, see csrc/mxq_check.cuh); same kernels otherwise
CHECKED_LIB_PATH = PKG / "libmxq_checked.so"
CHECKED_FLAGS = ["-DMXQ_DEBUG_BOUNDS=1"]

SOURCES = ["mxq_dual.cu", "mxq_compose.cu", "mx9.cu", "mx_packed.cu", "mx_cols_tma.cu", "mxq_mma_check.cu",
           "mxq_abi.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-diag-suppress", "177", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def _fingerprint(extra=()) -> str:
    h = hashlib.sha256()
    for f in sorted(list(CSRC.glob("*")) + list(INCLUDE.glob("*.h"))):
        if f.is_file():
            h.update(f.name.encode())
            h.update(f.read_bytes())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra)).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build_library(force: bool = False, verbose: bool = False, checked: bool = False) -> Path:
    """Build libmxq.so, or with `checked` the bounds-checked libmxq_checked.so."""
    extra = CHECKED_FLAGS if checked else []
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_dir = BUILD_DIR / "checked" if checked else BUILD_DIR
    stamp = build_dir / (lib_path.stem + ".stamp")
    fp = _fingerprint(extra)
    if not force and lib_path.exists() and stamp.exists() and stamp.read_text() == fp:
        return lib_path
    build_dir.mkdir(parents=True, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> Path:
        obj = build_dir / (src + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path.with_name(f".libmxq.{os.getpid()}.so")
    subprocess.run([cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *map(str, objs), "-o", str(tmp)],
                   check=True)
    os.replace(tmp, lib_path)
    stamp.write_text(fp)
    return lib_path


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
