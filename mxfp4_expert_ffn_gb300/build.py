"""Builds the CUDA library in-tree: csrc/*.cu -> libmoe_ffn.so (sm_103a only).

Each translation unit compiles in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -lineinfo -O3``; the objects go
to ``_build/`` next to this file and are relinked only when a source or
header changed.
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
OUT = os.path.join(HERE, "libmoe_ffn.so")
BUILD = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_ffn.so")


def _deps() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "moe_ffn.h")])


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, headers: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    if _stale(obj, [src] + headers):
        cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj + ".tmp"]
        subprocess.check_call(cmd)
        os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = [d for d in _deps() if not d.endswith(".cu")]
    if force:
        for o in glob.glob(os.path.join(BUILD, "*.o")):
            os.remove(o)
    if not force and not _stale(OUT, _deps()):
        return OUT
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, headers), srcs))
    tmp = OUT + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"])
    os.replace(tmp, OUT)
    return OUT


def build_synth(force: bool = False) -> str:
    """The GPU bank filler of the seeded input generators (synth/fill.cu)."""
    src = os.path.join(ROOT, "synth", "fill.cu")
    out = os.path.join(ROOT, "synth", "libsynth_cuda.so")
    if force or _stale(out, [src]):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc(), *ARCH, "-O3", "-Xcompiler", "-fPIC", "-shared", "-o", tmp,
                               src, "-lcudart"])
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
    print(build_synth(force=True))
