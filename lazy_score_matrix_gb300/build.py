"""Build libtp.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

Usage: ``python -m lazy_score_matrix_gb300.build`` (or ``__graft_entry__.build()``).
Objects go to ``lazy_score_matrix_gb300/_build/``; the library to ``lazy_score_matrix_gb300/libtp.so``.
A translation unit is recompiled when it or any header in csrc/ or include/ is newer than its object.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtp.so")
# calibration library of the benchmark (measured fp32 / fp64 FMA and exp2 rates), not part of libtp
PEAKS_SRC = os.path.join(PKG, "peaks", "tp_peaks.cu")
PEAKS_LIB = os.path.join(PKG, "libtp_peaks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libtp")


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, extra: list[str]) -> tuple[str, int, str]:
    obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return obj, r.returncode, (r.stdout + r.stderr)


def build(force: bool = False, jobs: int | None = None, verbose: bool = False, extra: list[str] | None = None) -> str:
    os.makedirs(OBJ_DIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr = _headers_mtime()
    todo = []
    for s in srcs:
        obj = os.path.join(OBJ_DIR, os.path.basename(s)[:-3] + ".o")
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(s), hdr):
            todo.append(s)
    jobs = jobs or max(1, min(len(todo) or 1, os.cpu_count() or 4))
    errors = []
    if todo:
        with cf.ThreadPoolExecutor(jobs) as ex:
            for obj, rc, out in ex.map(lambda s: _compile(s, extra or []), todo):
                if rc != 0:
                    errors.append((obj, out))
                elif verbose and out.strip():
                    print(out)
    if errors:
        for obj, out in errors:
            sys.stderr.write(f"--- {os.path.basename(obj)} ---\n{out[-4000:]}\n")
        raise RuntimeError(f"libtp build failed in {len(errors)} translation unit(s)")
    if force or not os.path.exists(PEAKS_LIB) or os.path.getmtime(PEAKS_LIB) < os.path.getmtime(PEAKS_SRC):
        tmp = PEAKS_LIB + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc(), *ARCH, "-O3", "-Xcompiler", "-fPIC", "-shared", "-o", tmp, PEAKS_SRC],
                           capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("libtp_peaks build failed")
        os.replace(tmp, PEAKS_LIB)
    objs = [os.path.join(OBJ_DIR, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if todo or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("libtp link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
