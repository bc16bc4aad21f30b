"""Builds libmoe.so in-tree with nvcc for sm_103a.

    python -m combine_router_gemm_top_b300.build

The library is the product's compute path: every kernel of the MoE layer
lives in csrc/ and is reached through the C ABI of include/moe.h.
"""
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmoe.so")
SOURCES = ["api.cu", "route.cu", "layout.cu", "permute_combine.cu",
           "grouped_ffn.cu", "layout_noalloc.cu", "router_stats.cu",
           "dispatch_extras.cu", "backward.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def headers():
    """Every header under csrc/: a change to any of them rebuilds the
    library (each translation unit may include any header)."""
    return sorted(os.path.basename(p) for ext in ("*.cuh", "*.h")
                  for p in glob.glob(os.path.join(CSRC, ext)))


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + headers()]
    deps.append(os.path.join(ROOT, "include", "moe.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=True, jobs=None):
    if not force and not _stale():
        return LIB
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    objs = []
    procs = []
    for src in SOURCES:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append(subprocess.Popen(cmd))
    for p in procs:
        if p.wait() != 0:
            raise RuntimeError("nvcc failed")
    tmp = LIB + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", *objs, "-o", tmp, "-lcudart"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv)
