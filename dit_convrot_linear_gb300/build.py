"""Build ``libtq.so`` (the CUDA library behind ``include/tq.h``) in-tree.

Each ``csrc/*.cu`` is compiled for sm_103a in parallel, then linked into one
shared library against the shared CUDA runtime (so the process's one
``libcudart`` serves both PyTorch and this library).  Run as a script or call
``build()``.  No cmake; the whole build takes well under two minutes.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link ``libtq.so``; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def build_variant(tag: str, defines, sources) -> str:
    """A copy of the library for the library's own tests: ``sources`` (file
    names under csrc/) recompiled with ``defines`` (NAME=VALUE strings) and
    linked with the regular objects of the other files.  Written to
    _build/libtq_<tag>.so; the product library is left as it is."""
    build()
    if not all(os.path.exists(os.path.join(OBJ_DIR, os.path.basename(x)[:-3] + ".o")) for x in _sources()):
        build(force=True)
    vdir = os.path.join(OBJ_DIR, tag)
    os.makedirs(vdir, exist_ok=True)
    flags = [f"-D{d}" for d in defines]
    objs = []
    for src in _sources():
        name = os.path.basename(src)
        if name in sources:
            obj = os.path.join(vdir, name[:-3] + ".o")
            cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *flags, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {name} ({tag}):\n{r.stdout}\n{r.stderr}")
            objs.append(obj)
        else:
            objs.append(os.path.join(OBJ_DIR, name[:-3] + ".o"))
    out = os.path.join(OBJ_DIR, f"libtq_{tag}.so")
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", out, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed ({tag}):\n{r.stdout}\n{r.stderr}")
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
