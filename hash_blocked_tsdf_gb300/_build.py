"""Builds the package's native libraries in-tree.

* ``libtsdf.so``: the CUDA integrate path behind the C ABI declared in
  ``include/tsdf.h`` (nvcc, sm_103a only, no fast-math, no FMA contraction).
* ``libscene_raycast.so``: the C ray caster that synthesises input frames.

Both are compiled from source on the machine that uses them (the x86 build
box cross-compiles the CUDA code; the Arm GPU host rebuilds everything).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")

CUDA_SOURCES = ["tsdf_volume.cu", "tsdf_alloc.cu", "tsdf_update.cu", "tsdf_extract.cu", "tsdf_table.cu",
                "tsdf_noalloc.cu"]
CUDA_HEADERS = ["tsdf_device.cuh", "tsdf_internal.h"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    # bit-exact voxel selection: IEEE division and square root, no fused
    # multiply-add contraction, no flush-to-zero
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtsdf.so")


def cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))


def tsdf_library_path() -> str:
    return os.path.join(PKG_DIR, "libtsdf.so")


def peaks_library_path() -> str:
    return os.path.join(PKG_DIR, "libtsdf_peaks.so")


def scene_library_path() -> str:
    return os.path.join(PKG_DIR, "libscene_raycast.so")


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + proc.stdout)
    return proc.stdout


def _newer(target, sources):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(s) <= t for s in sources)


def build_scene_library(force: bool = False) -> str:
    src = os.path.join(PKG_DIR, "scene_raycast.c")
    out = scene_library_path()
    if force or not _newer(out, [src]):
        tmp = out + f".tmp{os.getpid()}"
        _run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def build_tsdf_library(force: bool = False, extra_flags=(), verbose_ptxas: bool = False) -> str:
    out = tsdf_library_path()
    srcs = [os.path.join(CSRC, s) for s in CUDA_SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in CUDA_HEADERS] + [os.path.join(INCLUDE, "tsdf.h")]
    if not force and not extra_flags and not verbose_ptxas and _newer(out, deps):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    flags = NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC] + list(extra_flags)
    if verbose_ptxas:
        flags = flags + ["-Xptxas", "-v"]
    objs = []
    cmds = []
    for s in srcs:
        o = os.path.join(BUILD_DIR, os.path.basename(s) + ".o")
        objs.append(o)
        cmds.append([nvcc()] + flags + ["-c", s, "-o", o])
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        logs = list(ex.map(_run, cmds))
    tmp = out + f".tmp{os.getpid()}"
    # cudart is linked statically so the library loads without any search-path
    # setup; it still shares the process's CUDA context with PyTorch
    _run([nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "static",
          "-Xcompiler", "-fPIC", "-o", tmp] + objs)
    os.replace(tmp, out)
    if verbose_ptxas:
        print("".join(logs))
    return out


def build_peaks_library(force: bool = False) -> str:
    """The L2 reduction-throughput probe used by the benchmark."""
    src = os.path.join(CSRC, "peaks.cu")
    out = peaks_library_path()
    if force or not _newer(out, [src]):
        tmp = out + f".tmp{os.getpid()}"
        _run([nvcc()] + NVCC_FLAGS + ["-shared", "-cudart", "static", "-o", tmp, src])
        os.replace(tmp, out)
    return out


def build_all(force: bool = False) -> None:
    with concurrent.futures.ThreadPoolExecutor(max_workers=3) as ex:
        futs = [ex.submit(build_scene_library, force), ex.submit(build_tsdf_library, force),
                ex.submit(build_peaks_library, force)]
        for f in futs:
            f.result()
