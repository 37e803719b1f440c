"""Build libkda.so in-tree for sm_103a (nvcc for the kernels, g++ for the host code), and
the test-only libkda_selftest.so (tensor-core descriptor self-test; only the GPU tests load it).

Translation units compile in parallel; the results land in kda_state_chunked_gb300/_build/.
Usage: python -m kda_state_chunked_gb300.build [--force]
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
SO = os.path.join(BUILD, "libkda.so")
SELFTEST_SO = os.path.join(BUILD, "libkda_selftest.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CU_SOURCES = ["kernels/ckpt_copy.cu", "kernels/ckpt_q8.cu", "kernels/decode.cu", "kernels/prefill_simt.cu",
              "kernels/prefill_tc.cu", "kernels/prefill_split.cu", "host/tensor_map.cu",
              "host/prefill_noalloc.cu"]
SELFTEST_CU = ["selftest/tc_selftest.cu"]
CPP_SOURCES = ["host/pool.cpp", "host/split_plan.cpp", "host/api.cpp"]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: the KDA library needs the CUDA toolkit to build")


def _sources_mtime() -> float:
    t = os.path.getmtime(os.path.join(INCLUDE, "kda.h"))
    for dp, _, fs in os.walk(CSRC):
        for f in fs:
            t = max(t, os.path.getmtime(os.path.join(dp, f)))
    return max(t, os.path.getmtime(__file__))


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(SO) and os.path.exists(SELFTEST_SO)
            and min(os.path.getmtime(SO), os.path.getmtime(SELFTEST_SO)) >= _sources_mtime()):
        return SO
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    inc = ["-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in CU_SOURCES + SELFTEST_CU:
        obj = os.path.join(BUILD, src.replace("/", "_") + ".o")
        jobs.append([nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xptxas", "-v" if verbose else "-O3", *inc, "-c", os.path.join(CSRC, src),
                     "-o", obj])
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src.replace("/", "_") + ".o")
        jobs.append(["g++", "-O2", "-fPIC", "-std=c++17", "-Wall", "-I",
                     os.path.join(cuda, "include"), *inc, "-c", os.path.join(CSRC, src), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        outs = list(ex.map(_run, jobs))
    if verbose:
        for o in outs:
            if o.strip():
                print(o)
    obj_of = {src: os.path.join(BUILD, src.replace("/", "_") + ".o") for src in CU_SOURCES + SELFTEST_CU + CPP_SOURCES}
    for so, srcs in ((SO, CU_SOURCES + CPP_SOURCES), (SELFTEST_SO, SELFTEST_CU + ["host/tensor_map.cu"])):
        tmp = so + f".tmp{os.getpid()}"
        _run([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[obj_of[x] for x in srcs]])
        os.replace(tmp, so)
    return SO


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
