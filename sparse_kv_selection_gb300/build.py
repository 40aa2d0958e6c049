"""Build libprhs.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each translation unit compiles in parallel with nvcc; the objects link into
one shared library next to this file. Usage: ``python -m
sparse_kv_selection_gb300.build [--verbose]`` or ``build()`` from Python.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libprhs.so")
SOURCES = ["api.cu", "score.cu", "cis.cu", "attn.cu", "attn_cluster.cu", "select.cu", "retrieve.cu", "dense.cu",
           "noalloc.cu", "mass.cu", "grow.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "--expt-relaxed-constexpr", "-I", os.path.join(HERE, "..", "include")]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(src_files, target) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in src_files)


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile (if stale) and return the path of libprhs.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(HERE, "..", "include", "prhs.h"))
    if not force and not _stale(deps, LIB):
        return LIB
    cc = nvcc()

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *_flags(verbose), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, force="--force" in sys.argv))
