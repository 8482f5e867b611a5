"""Build libmla.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object file,
then all are linked into mla_absorbed_latent_gb300/lib/libmla.so against the
shared CUDA runtime (the one PyTorch already loaded).
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
OUT_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(OUT_DIR, "libmla.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing",
                     "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, obj: str, verbose_ptxas: bool) -> str:
    cmd = [nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build_library(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile every csrc/*.cu and link libmla.so; returns the library path."""
    srcs = sources()
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(ROOT, "include", "mla.h"))
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in srcs + hdrs)
        if os.path.getmtime(LIB) >= newest:
            return LIB
    objdir = os.path.join(OUT_DIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    objs = [os.path.join(objdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    logs = {}
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        futs = {ex.submit(_compile, s, o, verbose_ptxas): s for s, o in zip(srcs, objs)}
        for f in cf.as_completed(futs):
            logs[os.path.basename(futs[f])] = f.result()
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose_ptxas:
        for name in sorted(logs):
            sys.stderr.write(f"== {name}\n{logs[name]}")
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
