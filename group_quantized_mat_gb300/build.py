"""Builds the CUDA library libqmv.so in-tree (group_quantized_mat_gb300/_build/).

nvcc for sm_103a only (-gencode arch=compute_103a,code=sm_103a), one
translation unit per (bits, group_size) kernel table, compiled in parallel;
the codec is plain C++ (g++). The CUDA runtime is linked statically and the
library has no torch dependency. Usage: ``python -m group_quantized_mat_gb300.build``.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libqmv.so")
INCLUDE = os.path.join(ROOT, "include")

CU_SOURCES = ["qmv_api.cu", "qmv_noalloc.cu", "qmv_mx.cu", "qmv_inst_b4g64.cu", "qmv_inst_b4g128.cu", "qmv_inst_b2g64.cu", "qmv_inst_b2g128.cu"]
CXX_SOURCES = ["qmv_codec.cpp"]
HEADERS = ["qmv_plan.h", "qmv_kernel.cuh", "qmv_launch.cuh", "qmv_launch_decl.h"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "--fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def build(verbose: bool = False, extra_defines: tuple[str, ...] = (), out: str | None = None,
          force: bool = False) -> str:
    """Compile (if stale) and return the path of libqmv.so.

    ``extra_defines`` (e.g. ``("QMV_TEST_MUTATE_ORDER=1",)``) builds a variant
    into ``out`` -- used only by tests.
    """
    lib = out or LIB
    tag = "" if not extra_defines else "_" + "_".join(d.replace("=", "") for d in extra_defines)
    obj_dir = os.path.join(OUT_DIR, "obj" + tag)
    os.makedirs(obj_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "qmv.h")]
    nvcc = _nvcc()
    defs = [f"-D{d}" for d in extra_defines]
    jobs = []
    objs = []
    for src in CU_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append([nvcc, *NVCC_FLAGS, *defs, "-I", INCLUDE, "-I", CSRC, "-c", s, "-o", o])
    for src in CXX_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", *defs, "-I", INCLUDE,
                         "-c", s, "-o", o])
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for f in [ex.submit(_run, j) for j in jobs]:
                f.result()
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        _run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs,
              "-lpthread", "-ldl", "-lrt"])
        os.replace(tmp, lib)
    if verbose:
        print(lib)
    return lib


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)
