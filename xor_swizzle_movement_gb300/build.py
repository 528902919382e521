"""Build libswz.so (the CUDA library) in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process, in parallel, then one
link step makes the shared library.  Outputs land in
xor_swizzle_movement_gb300/_build/ (git-ignored).  No cmake, no torch build
machinery: the library's ABI is plain C (include/swz.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "_build", "libswz.so")
SOURCES = ["swz_abi.cu", "swz_relayout.cu", "swz_relayout_neg.cu", "swz_transpose.cu", "swz_bank.cu", "swz_tma.cu",
           "swz_tma_relayout.cu", "swz_probe.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
            f"-I{INCLUDE}", f"-I{CSRC}", *extra]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "swz.h"))
    cc = nvcc()
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or ptxas_info or _stale(o, [s, *headers]):
            extra = ["-Xptxas", "-v"] if ptxas_info else []
            jobs.append((src, [cc, *_flags(extra), "-c", s, "-o", o]))
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]

    def run(job):
        name, cmd = job
        if verbose:
            print(" ".join(cmd), flush=True)
        p = subprocess.run(cmd, capture_output=True, text=True)
        return name, p.returncode, p.stdout + p.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for name, rc, out in ex.map(run, jobs):
            if out and (verbose or ptxas_info or rc != 0):
                print(f"--- {name}\n{out}", file=sys.stderr)
            if rc != 0:
                raise RuntimeError(f"nvcc failed on {name}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv, force="--force" in sys.argv)
    print(LIB)
