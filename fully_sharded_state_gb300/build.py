"""Build the shard engine's CUDA library in-tree.

Compiles ``csrc/fsdp_kernels.cu`` (nvcc, sm_103a) and ``csrc/fsdp_capi.cpp``
(g++) in parallel and links ``_lib/libfsdp_shard.so`` with the CUDA runtime
linked statically. No cmake, no torch extension machinery: the library has a
plain C ABI (``include/fsdp_shard.h``).

    python -m fully_sharded_state_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(REPO, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libfsdp_shard.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["fsdp_kernels.cu", "fsdp_capi.cpp"]
HEADERS = [os.path.join(CSRC, "fsdp_internal.h"), os.path.join(INCLUDE, "fsdp_shard.h")]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(_cuda_home(), "bin", "nvcc")


def compile_commands(ptxas_verbose: bool = False) -> dict:
    cuda_inc = os.path.join(_cuda_home(), "include")
    inc = ["-I", INCLUDE, "-I", CSRC]
    cmds = {}
    cu = os.path.join(CSRC, "fsdp_kernels.cu")
    cmds[cu] = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                "-Xcompiler", "-fPIC,-ffp-contract=off", *inc, "-c", cu,
                "-o", os.path.join(BUILD, "fsdp_kernels.o")]
    if ptxas_verbose:
        cmds[cu].insert(1, "-Xptxas=-v")
    cpp = os.path.join(CSRC, "fsdp_capi.cpp")
    cmds[cpp] = ["g++", "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-Wall", *inc,
                 "-I", cuda_inc, "-c", cpp, "-o", os.path.join(BUILD, "fsdp_capi.o")]
    return cmds


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link the library if any source changed; returns its path."""
    if not force and not ptxas_verbose and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    cmds = compile_commands(ptxas_verbose)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, res

    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        results = list(ex.map(run, cmds.values()))
    for cmd, res in results:
        if verbose or ptxas_verbose:
            sys.stdout.write(res.stdout)
            sys.stderr.write(res.stderr)
        if res.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp,
            os.path.join(BUILD, "fsdp_kernels.o"), os.path.join(BUILD, "fsdp_capi.o")]
    if verbose:
        print(" ".join(link), flush=True)
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose))
