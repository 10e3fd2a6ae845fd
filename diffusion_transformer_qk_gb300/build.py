"""Build libqknr.so in-tree with nvcc for sm_103a.

The translation units compile in parallel; ptxas resource usage (registers,
stack frame, spill bytes, shared memory) of every kernel instance is kept
in ``_build/ptxas.log`` beside the objects.  ``--checked`` builds the debug
library libqknr_checked.so instead: the same sources compiled with
-DQKNR_CHECKED, whose kernels test every global access against the span of
its buffer and every shared-memory stage read against its stage, skip an
access that misses, and report QKNR_ERR_BOUNDS in the caller's status word.  A content stamp of the sources
and flags decides whether a rebuild is needed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libqknr.so"
CHECKED_LIB_NAME = "libqknr_checked.so"

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
CXX_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
             "-I" + INCLUDE, "-I" + CSRC]

SOURCES = [
    "qknr_api.cu",
    "qknr_host_api.cu",
    "qknr_inst_bf16_f32.cu",
    "qknr_inst_bf16_bf16.cu",
    "qknr_inst_fp16_f32.cu",
    "qknr_inst_fp16_bf16.cu",
    "adaln_api.cu",
    "adaln_inst.cu",
    "gn_api.cu",
]


def library_path(checked: bool = False) -> str:
    """The regular library, or the checked build (every kernel access tested
    against its buffer's span, QKNR_ERR_BOUNDS on a miss)."""
    return os.path.join(PKG, CHECKED_LIB_NAME if checked else LIB_NAME)


def _build_dir(checked: bool) -> str:
    return BUILD_DIR + ("_checked" if checked else "")


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqknr.so")
    return cand


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")


def _inputs() -> List[str]:
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh", ".h"))]
    files.extend(os.path.join(INCLUDE, f) for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h"))
    files.append(os.path.abspath(__file__))
    return files


def _flags(checked: bool) -> List[str]:
    return CXX_FLAGS + (["-DQKNR_CHECKED"] if checked else [])


def _stamp(checked: bool = False) -> str:
    h = hashlib.sha256()
    for f in _inputs():
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH_FLAGS + _flags(checked)).encode())
    return h.hexdigest()


def _stamp_path(checked: bool = False) -> str:
    return os.path.join(_build_dir(checked), "stamp")


def is_stale(checked: bool = False) -> bool:
    if not os.path.exists(library_path(checked)) or not os.path.exists(_stamp_path(checked)):
        return True
    with open(_stamp_path(checked)) as f:
        return f.read().strip() != _stamp(checked)


def build_library(verbose: bool = False, jobs: int = 0, checked: bool = False) -> str:
    """Compile every translation unit and link libqknr.so (with ``checked``,
    libqknr_checked.so, built with -DQKNR_CHECKED); returns its path."""
    bdir = _build_dir(checked)
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    objs, cmds = [], []
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([cc, *ARCH_FLAGS, *_flags(checked), "-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        return subprocess.run(cmd, capture_output=True, text=True)

    with ThreadPoolExecutor(max_workers=jobs or len(cmds)) as ex:
        results = list(ex.map(run, cmds))
    log = []
    for cmd, r in zip(cmds, results):
        log.append("$ " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    with open(os.path.join(bdir, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    out = library_path(checked)
    tmp = out + ".tmp"
    link = [cc, *ARCH_FLAGS, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", "-rpath," + cuda_lib_dir()]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"linking {os.path.basename(out)} failed")
    os.replace(tmp, out)
    with open(_stamp_path(checked), "w") as f:
        f.write(_stamp(checked))
    if verbose:
        print("\n".join(log))
    return out


def ensure_built(checked: bool = False) -> str:
    if is_stale(checked):
        build_library(checked=checked)
    return library_path(checked)


if __name__ == "__main__":
    chk = "--checked" in sys.argv
    build_library(verbose="-v" in sys.argv, checked=chk)
    print(library_path(chk))
