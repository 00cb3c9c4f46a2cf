"""Build libmk.so in-tree for sm_103a (nvcc, one -gencode, translation units in parallel)."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmk.so")
SOURCES = ["mk_abi.cu", "mk_kernels.cu", "mk_noalloc.cu", "mk_attention.cu"]
HEADERS = ["mk_internal.h", "mk_ptx.cuh", "mk_device.cuh"]
GENCODE = "arch=compute_103a,code=sm_103a"


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "mk.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA sources and link libmk.so next to this file; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = [nvcc, "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xptxas", "-v", f"-I{INCLUDE}", f"-I{CSRC}"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD_DIR, src.replace(".cu", ".ptxas.log")), "w")
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
        objs.append(obj)
    failed = []
    for src, pr, log in procs:
        rc = pr.wait()
        log.close()
        if rc != 0:
            failed.append(src)
    if failed:
        for src in failed:
            sys.stderr.write(open(os.path.join(BUILD_DIR, src.replace(".cu", ".ptxas.log"))).read())
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-shared", "-gencode", GENCODE, "-o", tmp] + objs)
    os.replace(tmp, LIB)
    if verbose:
        for src in SOURCES:
            sys.stdout.write(open(os.path.join(BUILD_DIR, src.replace(".cu", ".ptxas.log"))).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
