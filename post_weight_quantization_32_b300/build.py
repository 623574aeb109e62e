"""Build libawq.so in-tree with nvcc for sm_103a (B300).

    python post_weight_quantization_32_b300/build.py [-v] [-f]

Each .cu file under csrc/ is compiled to an object in _build/ (skipped when
up to date), then linked into post_weight_quantization_32_b300/libawq.so with
the CUDA runtime linked statically.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libawq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-Xptxas", "-v",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


# The search and tensor-core clipping kernels split their registers between
# warpgroups with setmaxnreg (128 threads x 48 + 256 threads x 200 + 128
# threads x 56 or 64); that split must fit in what the block is launched
# with, so every such kernel has to be compiled to the full 128 registers a
# thread that its launch bounds allow.
SEARCH_KERNEL_REGS = 128


def _check_registers(src: str, text: str) -> None:
    current = None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current and ("awq_search_kernel" in current or "clip_mma_kernel" in current):
            if int(m.group(1)) != SEARCH_KERNEL_REGS:
                raise RuntimeError("%s: %s compiled to %s registers, the register split needs %d"
                                   % (os.path.basename(src), current, m.group(1), SEARCH_KERNEL_REGS))
            current = None


def _compile(src: str, obj: str, log: list) -> None:
    cmd = [_nvcc()] + ARCH + FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log.append((src, r.stdout + r.stderr))
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (os.path.basename(src), r.stdout + r.stderr))
    try:
        _check_registers(src, r.stdout + r.stderr)
    except RuntimeError:
        os.remove(obj)
        raise


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    dep_t = _deps_mtime()
    jobs, objs, log = [], [], []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), dep_t):
            jobs.append((s, o))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(lambda j: _compile(j[0], j[1], log), jobs))
    if jobs or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        # cuBLAS serves GPTQ's plain GEMMs (dynamic: the CUDA toolkit's libcublas)
        cmd = [_nvcc()] + ARCH + ["-shared", "--cudart", "static", "-o", LIB] + objs + ["-lcublas"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    if verbose:
        for src, out in log:
            print("==", os.path.basename(src))
            print(out)
    return LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, force="-f" in sys.argv)
    print(LIB)
