"""Build the CUDA libraries in-tree for sm_103a (GB300).

    python -m bit_expert_ffn_gb300.build

* ``libmoe_gb300.so``  -- the product: every ``csrc/*.cu`` except the input
  generator, C ABI declared in ``include/moe_gb300.h``.
* ``libmoe_synth.so``  -- the device-side seeded input generator
  (``csrc/synth_fill.cu``), kept apart from the product library.

Translation units compile in parallel; a unit is rebuilt only when it or a
header changed.  Objects go to ``_build/`` next to this file.
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
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_gb300.so")
SYNTH_LIB = os.path.join(HERE, "libmoe_synth.so")
SYNTH_SRC = "synth_fill.cu"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build the library")
    return path


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra=()) -> str:
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    if extra or _stale(obj, [src] + _headers() + [__file__]):
        cmd = [nvcc()] + NVFLAGS + list(extra) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if r.stderr.strip():
            sys.stderr.write(r.stderr)
    return obj


def _link(objs, out):
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-Xlinker", "-rpath", "-Xlinker", "/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {out} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(verbose_ptxas: bool = False) -> tuple[str, str]:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = dict(zip(srcs, ex.map(lambda s: _compile(s, extra), srcs)))
    prod = [o for s, o in objs.items() if os.path.basename(s) != SYNTH_SRC]
    syn = [o for s, o in objs.items() if os.path.basename(s) == SYNTH_SRC]
    if _stale(LIB, prod):
        _link(prod, LIB)
    if syn and _stale(SYNTH_LIB, syn):
        _link(syn, SYNTH_LIB)
    return LIB, SYNTH_LIB


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
