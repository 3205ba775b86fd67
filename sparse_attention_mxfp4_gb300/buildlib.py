"""Build the scorer's CUDA library (libmx4index.so) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libmx4index.so")
SOURCES = ["mx4_index.cu"]
HEADER = os.path.join(ROOT, "include", "mx4_index.h")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def source_files() -> list[str]:
    """Every file the library is compiled from: all of csrc/ (.cu and .cuh),
    the public header and this script."""
    files = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")))
    return files + [HEADER, os.path.abspath(__file__)]


def source_digest(extra_flags=()) -> str:
    """SHA-256 over the contents of every source file and the nvcc flags."""
    h = hashlib.sha256()
    for f in source_files():
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join([*NVCC_FLAGS, *extra_flags]).encode())
    return h.hexdigest()


def _stamp(lib_path: str) -> str:
    return lib_path + ".sha256"


def _stale(lib_path: str = LIB_PATH, extra_flags=()) -> bool:
    """True unless the library exists and was built from exactly the current
    sources (content digest recorded beside it at build time)."""
    if not os.path.exists(lib_path) or not os.path.exists(_stamp(lib_path)):
        return True
    with open(_stamp(lib_path)) as fh:
        return fh.read().strip() != source_digest(extra_flags)


def build(force: bool = False, verbose: bool = False, lib_path: str = LIB_PATH, extra_flags=()) -> str:
    """Compile csrc/mx4_index.cu into ``lib_path`` (skipped when the recorded
    source digest matches).  ``extra_flags`` are appended to nvcc's flags."""
    if not force and not _stale(lib_path, extra_flags):
        return lib_path
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    digest = source_digest(extra_flags)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"),
           *[os.path.join(CSRC, s) for s in SOURCES], "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib_path)
    with open(_stamp(lib_path), "w") as fh:
        fh.write(digest + "\n")
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
