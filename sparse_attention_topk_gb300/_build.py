"""Builds libtks.so (the CUDA selection library) in-tree with nvcc, for sm_103a."""

from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtks.so")

SOURCES = [os.path.join(CSRC, "tks_select.cu"), os.path.join(CSRC, "tks_select512.cu"),
           os.path.join(CSRC, "tks_order.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "tks_device.cuh"), os.path.join(CSRC, "tks_kernel.cuh"),
                     os.path.join(CSRC, "tks_internal.h"), os.path.join(INCLUDE, "tks.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtks")
    return cand


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(s) <= t for s in DEPENDS)


# A measurement build: the first-round histogram with warp-aggregated adds
# (match_any) instead of plain shared-memory adds, otherwise the same library.
HIST_AGGREGATE_PATH = os.path.join(BUILD_DIR, "libtks_hist_aggregate.so")


def build(force: bool = False, verbose_ptxas: bool = False, out: str = LIB_PATH,
          hist_aggregate: bool = False) -> str:
    """Compile libtks.so unless it is newer than every source; returns its path.
    hist_aggregate: the measurement build (HIST_AGGREGATE_PATH by default)."""
    if hist_aggregate and out == LIB_PATH:
        out = HIST_AGGREGATE_PATH
    if not force and up_to_date(out):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tag = f".tmp{os.getpid()}"
    nvcc = nvcc_path()
    # one process per translation unit, in parallel, then one link
    objs = [os.path.join(os.path.dirname(out), os.path.basename(src) + tag + ".o") for src in SOURCES]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = [nvcc, *NVCC_FLAGS, f"-I{INCLUDE}", f"-I{CSRC}", "-c", src, "-o", obj]
        if hist_aggregate:
            cmd.insert(1, "-DTKS_HIST_AGGREGATE=1")
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd)))
    failed = [src for src, pr in procs if pr.wait() != 0]
    try:
        if failed:
            raise subprocess.CalledProcessError(1, f"nvcc -c {' '.join(failed)}")
        tmp = out + tag
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs,
                        "-o", tmp], check=True)
        os.replace(tmp, out)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
