"""Build of the CUDA library ``libmpgemm.so`` (in-tree, sm_103a only).

Every translation unit under ``csrc/`` is compiled by nvcc in parallel with
``-gencode arch=compute_103a,code=sm_103a`` and linked (static CUDA runtime)
into ``mixed_precision_matmul_gb300/_build/libmpgemm.so``.  The ptxas resource
report (``-Xptxas -v``: registers, spills, shared memory) of each unit is kept
in ``_build/ptxas.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmpgemm.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = [
    "api.cu",
    "host_common.cu",
    "plan.cu",
    "host_api.cu",
    "attention_api.cu",
    "acc_layout.cpp",
    "aux_kernels.cu",
    "ffma.cu",
    "tc_direct.cu",
    "tc_staged.cu",
    "tc_generic.cu",
    "prepass.cu",
    "tc_pair.cu",
    "attention.cu",
    "tmem_probe.cu",
]
HEADERS = ["ptx.cuh", "internal.h", "tc_gemm.cuh", "outio.cuh", "host.h", "staging.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libmpgemm")
    return cand


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> tuple[str, str]:
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src + ".o")
    deps = [path, os.path.join(INCLUDE, "mpgemm.h")] + [os.path.join(CSRC, h) for h in HEADERS]
    if not _stale(obj, deps):
        return obj, ""
    cmd = [_nvcc(), "-c", path, "-o", obj + ".tmp", "-std=c++17", "-O3", "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC] + ARCH
    if src.endswith(".cu"):
        cmd += ["-Xptxas", "-v", "--expt-relaxed-constexpr"]
    else:
        cmd += ["-x", "c++"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (when sources changed) and link libmpgemm.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
    jobs = min(len(SOURCES), max(2, os.cpu_count() or 2))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(_compile, SOURCES))
    objs = [o for o, _ in results]
    logs = "".join(f"== {s}\n{log}" for s, (_, log) in zip(SOURCES, results) if log)
    if logs:
        with open(os.path.join(BUILD, "ptxas.log"), "w") as fh:
            fh.write(logs)
    if _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
