"""Builds libprm.so in-tree: every CUDA source under csrc/ compiled for
sm_103a with nvcc (in parallel), linked into one shared library next to this
file. No cmake; incremental on source and header modification times."""
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
OBJDIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libprm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I" + INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libprm")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


# The source of each kernel family's kernels; every family also depends on
# the engine that plans and launches it (prm_api.cu) and on the headers.
FAMILY_SOURCES = {
    "ns_prep": ("refresh.cu",),
    "ns_gram": ("ns5_gemm.cu",),
    "ns_poly": ("ns5_gemm.cu",),
    "ns_sym": ("ns5_gemm.cu",),
    "ns_combine": ("ns5_gemm.cu",),
    "ns_small": ("ns_small.cu",),
    "rownorm_wide": ("rownorm.cu",),
    "rownorm_tall": ("rownorm.cu",),
}
_ENGINE = "prm_api.cu"


def _code_only(text: bytes) -> bytes:
    """The source without // and /* */ comments and blank-line differences,
    so that editing a comment leaves a digest unchanged. (The sources hold
    no comment markers inside string literals.)"""
    import re
    t = text.decode("utf-8")
    t = re.sub(r"/\*.*?\*/", "", t, flags=re.S)
    t = re.sub(r"//[^\n]*", "", t)
    lines = [ln.rstrip() for ln in t.splitlines()]
    return "\n".join(ln for ln in lines if ln).encode()


def source_digest(family: str) -> str:
    """sha256 over the code (comments stripped) of one kernel family's
    source, the engine and the headers: identifies the kernels and launch
    plan that a stored profile of that family was taken on."""
    import hashlib
    names = set(FAMILY_SOURCES[family]) | {_ENGINE}
    h = hashlib.sha256()
    for path in [p for p in _sources() if os.path.basename(p) in names] + _headers():
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(_code_only(f.read()))
    return h.hexdigest()[:16]


def build_library(verbose: bool = False, force: bool = False) -> str:
    """Compiles csrc/*.cu and links libprm.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(OBJDIR, exist_ok=True)
    headers = _headers()
    jobs = []
    for src in _sources():
        obj = os.path.join(OBJDIR, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, [src] + headers):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        return obj

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(compile_one, jobs))
    objs = [os.path.join(OBJDIR, os.path.basename(s)[:-3] + ".o") for s in _sources()]
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(verbose=True, force="--force" in sys.argv))
