"""Build libsage_gb300.so from csrc/ with nvcc for sm_103a (in-tree, no install step).

    python -m bit_trainable_attention_sage_gb300.build [--force] [--verbose]

Each translation unit compiles in parallel into _build/, then nvcc links the shared library next
to this file.  The build is skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsage_gb300.so")
# Test-only copy of the library for the timeout test: bounded waits of about 0.1 s, and a
# backward producer that never issues one Q^ block (SAGE_TEST_SKIP_Q_ARRIVAL), so that the waits
# for it run out and the call reports SAGE_ERR_TIMEOUT.  Never loaded by the product binding.
VARIANTS = {
    "faultsim": dict(lib=os.path.join(HERE, "libsage_gb300_faultsim.so"),
                     objdir=os.path.join(HERE, "_build_faultsim"),
                     defines=["-DSAGE_WAIT_CYCLES=200000000ull", "-DSAGE_TEST_SKIP_Q_ARRIVAL=1"]),
}
SOURCES = ["sage_quant.cu", "sage_fwd.cu", "sage_bwd.cu", "sage_capi.cu", "sage_noalloc.cu"]
HEADERS = ["sage_device.cuh", "sage_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libsage_gb300.so")
    return exe


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "sage.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str, verbose: bool, objdir: str = OBJDIR, defines=()) -> str:
    obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, variant: str | None = None) -> str:
    """Compile and link the library (or a test-only ``variant`` of it); returns its path."""
    lib, objdir, defines = LIB, OBJDIR, []
    if variant is not None:
        v = VARIANTS[variant]
        lib, objdir, defines = v["lib"], v["objdir"], v["defines"]
    if not force and up_to_date(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, objdir, defines), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
