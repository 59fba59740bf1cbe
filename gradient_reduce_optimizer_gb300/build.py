"""Build the C-ABI library ``libcc_dp.so`` in-tree for sm_103a (GB300).

Each CUDA translation unit is compiled by nvcc in parallel into ``_build/``
and linked into ``gradient_reduce_optimizer_gb300/libcc_dp.so`` with the
CUDA runtime linked statically and cuBLAS (used only by the overlap
measurement's proxy backward) dynamically.  Host code is built with
``-ffp-contract=off`` so the AdamW scalars computed on the host are single
binary32 roundings.  Run as a script, or call :func:`build`.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIBRARY = os.path.join(PKG, "libcc_dp.so")

SOURCES = ["cc_dp_kernels.cu", "cc_dp_bulk.cu", "cc_dp_unfused.cu", "cc_dp_api.cu",
           "cc_overlap.cu", "cc_tp.cu", "cc_tp_fused.cu"]
HEADERS = [os.path.join(CSRC, "cc_dp_internal.h"), os.path.join(CSRC, "cc_dp_device.cuh"),
           os.path.join(CSRC, "cc_trace.h"), os.path.join(INCLUDE, "cc_dp.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false",
    "-Xcompiler", "-fPIC,-fvisibility=hidden,-ffp-contract=off,-Wall",
    "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")


def cuda_lib_dirs() -> List[str]:
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    return [d for d in (os.path.join(home, "lib64"),
                        os.path.join(home, "targets", "sbsa-linux", "lib"),
                        os.path.join(home, "targets", "x86_64-linux", "lib"))
            if os.path.isdir(d)]


def _stale(target: str, deps: List[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False,
          extra_flags: List[str] = (), build_dir: str = BUILD_DIR,
          library: str = LIBRARY) -> str:
    """Compile (if stale) and link the library; returns its path.

    ``extra_flags`` (e.g. ``-DCC_DP_THREADS=512``) go to every nvcc call;
    give such builds their own ``build_dir`` and ``library`` path.
    """
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    objs, procs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [path, *HEADERS]):
            cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", path, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT,
                                                text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if force or procs or _stale(library, objs):
        rpath = ":".join(cuda_lib_dirs())
        tmp = library + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
               "-lcublas", "-lcublasLt", f"-Xlinker=-rpath={rpath}"]
        cmd += [f"-L{d}" for d in cuda_lib_dirs()]
        subprocess.run(cmd, check=True)
        os.replace(tmp, library)
    return library


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
