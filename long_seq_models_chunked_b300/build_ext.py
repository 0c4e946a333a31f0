"""Builds the C-ABI library in-tree with nvcc for sm_103a.

    python -m long_seq_models_chunked_b300.build_ext [-v]

Every .cu file under csrc/ is compiled to an object under _build/<variant>/
(in parallel), then linked with the static CUDA runtime into a shared library
that sits next to this file. The library exports only the extern "C" entry
points declared in include/ttt.h. Two variants are built from the same sources:

  libttt_b300.so        the tensor-core kernels share operand tiles across the
                        CTAs of a cluster by TMA multicast (one GPU per process)
  libttt_b300_local.so  built with TTT_NO_MULTICAST: clusters of one CTA, no
                        multicast and no CTA pairs; the library a process that
                        runs beside ranks on other GPUs loads

The environment variable TTT_B300_LIBRARY=local makes the Python binding load
the second one.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB_NAME = "libttt_b300.so"
LOCAL_LIB_NAME = "libttt_b300_local.so"
MC_LIB_PATH = os.path.join(PKG, LIB_NAME)
LOCAL_LIB_PATH = os.path.join(PKG, LOCAL_LIB_NAME)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]
VARIANTS = {
    "multicast": ([], MC_LIB_PATH),
    "local": (["-DTTT_NO_MULTICAST"], LOCAL_LIB_PATH),
}


def library_path() -> str:
    """The library the binding loads: the local variant when the environment
    asks for it (TTT_B300_LIBRARY=local), else the multicast one."""
    v = os.environ.get("TTT_B300_LIBRARY", "multicast")
    if v not in VARIANTS:
        raise ValueError(f"TTT_B300_LIBRARY={v!r}: expected one of {sorted(VARIANTS)}")
    return VARIANTS[v][1]


LIB_PATH = library_path()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _compile(src: str, outdir: str, flags, verbose: bool) -> str:
    obj = os.path.join(outdir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *flags, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr)
    return obj


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build(verbose: bool = False, extra=(), variants=tuple(VARIANTS)) -> str:
    """Compiles and links the requested variants; returns the path of the
    library the binding loads."""
    srcs = sources()
    jobs = []
    for v in variants:
        flags, _ = VARIANTS[v]
        outdir = os.path.join(BUILD, v)
        os.makedirs(outdir, exist_ok=True)
        jobs += [(v, s, outdir, [*flags, *extra]) for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(16, len(jobs))) as ex:
        objs = list(ex.map(lambda j: (j[0], _compile(j[1], j[2], j[3], verbose)), jobs))
    for v in variants:
        path = VARIANTS[v][1]
        tmp = path + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "--cudart", "static", "-o", tmp, *[o for vv, o in objs if vv == v]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({v}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)
    return library_path()


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
