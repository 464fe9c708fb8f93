"""Build libpsg.so (the C-ABI library) in-tree with nvcc for sm_103a.

Every translation unit compiles in parallel into ``_build/``; the shared
library lands next to this file.  Elementwise and reduction units are
compiled with IEEE division/sqrt, no flush-to-zero and no FMA contraction,
so each node of a program rounds exactly once, as a node of the op graph
does.  The contraction units may contract multiply-adds (their results are
bounded by the reduction-order term, not by per-node rounding).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(HERE, "libpsg.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
STRICT = ["-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false"]
# units whose float arithmetic is allowed to contract a*b+c into one FMA
FMA_OK = {"contract_simt.cu", "contract_tc.cu"}


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _deps_mtime():
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    hs.append(os.path.join(INCLUDE, "psg.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str) -> str:
    name = os.path.basename(src)
    obj = os.path.join(BUILD, name + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _deps_mtime()):
        return obj
    flags = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    flags += ARCH
    if name.endswith(".cu"):
        flags += [] if name in FMA_OK else STRICT
        flags += ["-Xptxas", "-v"] if os.environ.get("PSG_PTXAS_VERBOSE") else []
    cmd = [_nvcc(), "-c", src, "-o", obj + ".tmp"] + flags
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (name, " ".join(cmd), r.stderr))
    if os.environ.get("PSG_PTXAS_VERBOSE"):
        print(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, jobs: int | None = None) -> str:
    """Compile every unit under csrc/ and link libpsg.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    if force:
        for o in glob.glob(os.path.join(BUILD, "*.o")):
            os.remove(o)
    jobs = jobs or max(1, min(len(srcs), os.cpu_count() or 4))
    with cf.ThreadPoolExecutor(jobs) as ex:
        objs = list(ex.map(_compile, srcs))
    newest = max(os.path.getmtime(o) for o in objs)
    if force or not os.path.exists(SO) or os.path.getmtime(SO) < newest:
        tmp = SO + ".tmp%d" % os.getpid()
        cmd = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-lcudart_static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, SO)
    return SO


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv))
