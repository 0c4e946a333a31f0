"""The two builds of the library: the single-GPU build shares operand tiles
across the CTAs of a cluster with TMA multicast; the build that a process
running beside ranks on other GPUs loads contains no multicast instruction at
all (checked on the preprocessed sources, which is what the compiler sees), and
the multi-GPU benchmark refuses the multicast build."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from long_seq_models_chunked_b300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PTX_MULTICAST = "multicast::cluster"


def _preprocess(src, defines):
    cmd = [build_ext.nvcc(), *build_ext.ARCH, "-std=c++17", "--expt-relaxed-constexpr",
           "-I", os.path.join(ROOT, "include"), *defines, "-E", src]
    return subprocess.run(cmd, capture_output=True, text=True, check=True).stdout


def test_local_build_compiles_no_multicast_instruction():
    srcs = build_ext.sources()
    assert srcs
    for src in srcs:
        assert PTX_MULTICAST not in _preprocess(src, ["-DTTT_NO_MULTICAST"]), src
    # the multicast build does use it (so the check above can see it)
    tc = os.path.join(build_ext.CSRC, "ttt_tc.cu")
    assert PTX_MULTICAST in _preprocess(tc, [])


def test_only_one_header_spells_the_multicast_instructions():
    hits = []
    for f in glob.glob(os.path.join(build_ext.CSRC, "*")):
        if PTX_MULTICAST in open(f, errors="replace").read():
            hits.append(os.path.basename(f))
    assert hits == ["tc_ptx_mc.cuh"], hits


def test_feature_flags_of_the_two_builds():
    mc = ctypes.CDLL(build_ext.MC_LIB_PATH)
    local = ctypes.CDLL(build_ext.LOCAL_LIB_PATH)
    assert mc.ttt_build_features() & 1 == 1
    assert local.ttt_build_features() & 1 == 0


def test_multi_gpu_bench_refuses_the_multicast_build():
    import bench
    bench.check_library_for_world(1, 1)        # one GPU: either build
    bench.check_library_for_world(0, 4)        # several GPUs: the local build
    with pytest.raises(SystemExit, match="cluster multicast"):
        bench.check_library_for_world(1, 2)
