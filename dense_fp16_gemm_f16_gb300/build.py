"""Build libgemm_f16.so in-tree with nvcc for sm_103a.

The library is a plain shared object with a C ABI (include/gemm_f16.h); the
CUDA runtime is linked statically and its symbols are hidden, so the only
exported names are the gemm_* entry points.  Translation units compile in
parallel; a rebuild happens only when a source or header is newer than the
library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libgemm_f16.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

SOURCES = ["api.cu", "tiled_2cta.cu", "tiled_2cta512.cu", "tiled_1cta.cu", "skinny.cu", "streamk.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                           "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _inputs() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    lib_mtime = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > lib_mtime for p in _inputs())


def _run(cmd: list[str], verbose: bool) -> None:
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")
    if verbose and r.stdout.strip():
        print(r.stdout, flush=True)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          extra_flags=(), lib_path: str | None = None) -> str:
    """Compile the CUDA sources and link libgemm_f16.so; returns its path.

    ``extra_flags`` (e.g. ``["-DGEMM_GROUP_M=16"]``) and ``lib_path`` build a
    separately named copy with other compile-time settings; such builds always
    recompile and never replace the default library.
    """
    custom = bool(extra_flags) or lib_path is not None
    out = lib_path or LIB_PATH
    if not force and not ptxas_info and not custom and not is_stale():
        return out
    build_dir = BUILD_DIR if not custom else out + ".objs"
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + list(extra_flags)
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([cc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(lambda c: _run(c, verbose or ptxas_info), cmds))
    tmp = out + f".tmp{os.getpid()}"
    _run([cc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs, "-Xlinker", "--exclude-libs,ALL"], verbose)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB_PATH)
