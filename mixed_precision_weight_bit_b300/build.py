"""Builds libvbq.so in-tree for sm_103a with nvcc (no JIT cache, no torch extension).

Usage: python mixed_precision_weight_bit_b300/build.py [--force]
(run it by path: importing the package loads the library this script builds)
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(OUT_DIR, "libvbq.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
CUDA_LIB = "/usr/local/cuda/lib64"

SOURCES = ["pack.cpp", "plan.cpp", "gemv_plan.cpp", "kernels.cu", "gemm_tc.cu", "model.cu", "attention.cu", "quantize.cpp", "fakequant.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(os.path.dirname(HERE), "include", "vbq.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, defines=None, out_dir: str = OUT_DIR) -> str:
    """Compiles the sources and links <out_dir>/libvbq.so. defines: extra -D values for tuning builds."""
    lib = os.path.join(out_dir, "libvbq.so")
    if not force and out_dir == OUT_DIR and not defines and up_to_date():
        return LIB
    os.makedirs(out_dir, exist_ok=True)
    objs = []
    cmds = []
    dflags = [f"-D{d}" for d in (defines or [])]
    for src in SOURCES:
        obj = os.path.join(out_dir, src.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        lang = ["-x", "cu"] if src.endswith(".cu") else []
        cmds.append([NVCC, *GENCODE, *FLAGS, *dflags, *lang, "-c", os.path.join(CSRC, src), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        logs = list(ex.map(run, cmds))
    link = [NVCC, *GENCODE, "-shared", "-cudart", "shared", "-o", lib + ".tmp", *objs,
            "-Xlinker", f"-rpath,{CUDA_LIB}", "-Xlinker", "--no-undefined", "-L" + CUDA_LIB]
    logs.append(run(link))
    os.replace(lib + ".tmp", lib)
    if verbose:
        print("\n".join(l for l in logs if l.strip()))
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
