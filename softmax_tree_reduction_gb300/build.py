"""Build libtreeattn.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel, then linked into
``softmax_tree_reduction_gb300/libtreeattn.so`` (static CUDA runtime, no
torch headers).  Objects go to ``softmax_tree_reduction_gb300/_build/``.

``build(debug=True)`` makes the bounds-checking library instead,
``libtreeattn_debug.so`` (objects in ``_build_debug/``): the same sources
compiled with TA_DEBUG_BOUNDS, whose kernels check computed indices against
their buffers, skip an access that falls outside and report it through the
device error word (TA_ERR_DEVICE_BOUNDS).  Point the binding at it with the
TREE_ATTN_LIBRARY environment variable.

    python -m softmax_tree_reduction_gb300.build [--verbose-ptxas] [--force] [--debug]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtreeattn.so")
LIB_DEBUG = os.path.join(HERE, "libtreeattn_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["api.cu", "combine.cu", "split_kv_mma.cu", "split_kv_fma_bf16.cu", "split_kv_fma_f32.cu",
           "noalloc.cu", "split_kv_fp8.cu", "split_kv_tc05.cu", "split_kv_tc05_fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tree_attn.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date(lib: str = LIB) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime()


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    build_dir = BUILD + "_debug" if debug else BUILD
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if debug:
        extra.append("-DTA_DEBUG_BOUNDS")
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                                 text=True)))
    failed = []
    for src, cmd, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out))
        elif out and (verbose_ptxas or not quiet):
            sys.stdout.write(f"--- {src}\n{out}")
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = lib + ".tmp"
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt",
                    "-lpthread"], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv, quiet=False,
                debug="--debug" in sys.argv))
