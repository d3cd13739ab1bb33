"""Builds libmoe_ep.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process, in parallel, then one
link step produces ``_build/libmoe_ep.so`` next to this file. No fast-math:
the FP8 scales need IEEE division and the combine needs exact fma/round.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libmoe_ep.so")
# The same sources with device bounds checks (MOE_DEBUG_BOUNDS): every row
# index a kernel computes is checked against its buffer before the access.
DEBUG_LIB_PATH = os.path.join(BUILD_DIR, "libmoe_ep_debug.so")
SOURCES = ["api.cu", "layout.cu", "dispatch.cu", "combine.cu", "layout_noalloc.cu", "two_stage.cu",
           "fused.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
VARIANTS = {"release": ([], BUILD_DIR, LIB_PATH),
            "debug": (["-DMOE_DEBUG_BOUNDS"], os.path.join(BUILD_DIR, "debug"), DEBUG_LIB_PATH)}


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def up_to_date(variant: str = "release") -> bool:
    lib = VARIANTS[variant][2]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False,
          variants=("release", "debug")) -> str:
    """Compiles every translation unit of every requested variant in parallel
    (one nvcc process each), then links one library per variant. Returns the
    release library's path."""
    todo = [v for v in variants if force or not up_to_date(v)]
    if not todo:
        return LIB_PATH
    base = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
            *ARCH]
    if ptxas_v:
        base += ["-Xptxas", "-v"]
    procs = []
    objs = {}
    for v in todo:
        defs, odir, _ = VARIANTS[v]
        os.makedirs(odir, exist_ok=True)
        for src in SOURCES:
            obj = os.path.join(odir, src.replace(".cu", ".o"))
            objs.setdefault(v, []).append(obj)
            cmd = [nvcc(), *base, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((f"{v}:{src}",
                          subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for name, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(f"{name}:\n{text}")
        elif text.strip() and (verbose or ptxas_v):
            print(text, file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    for v in todo:
        lib = VARIANTS[v][2]
        tmp = lib + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc(), "-shared", *ARCH, "-o", tmp, *objs[v], "-lcudart"])
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="-v" in sys.argv))
