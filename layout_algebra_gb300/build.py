"""Build the native library ``libgb300gemm.so`` in-tree.

One shared library holds the host layout library (C++17), the sm_103a kernels and both
C ABIs (include/gb300_gemm.h, include/layout_algebra.h).  Objects compile in parallel
(the kernel instances in INST_GROUPS compilations of gemm_inst.cu);
the CUDA runtime is linked statically and the driver's tensor-map encoder is looked up
at run time, so the library loads on hosts without a GPU driver.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgb300gemm.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["layout.cpp", "layout_capi.cpp", "host_staging.cpp", "gemm_sm103.cu", "gemm_inst.cu"]
HEADERS = ["layout.hpp", "ptx.cuh", "gemm_kernel.cuh", "gemm_launch.cuh"]
INST_GROUPS = 14   # GB_INST_GROUP values of gemm_inst.cu
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _deps():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, h) for h in os.listdir(INCLUDE) if h.endswith(".h")]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _jobs():
    """(source, object name, extra flags) of every object of the library."""
    jobs = []
    for s in SOURCES:
        if s == "gemm_inst.cu":
            jobs += [(s, "gemm_inst_%d.o" % g, ["-DGB_INST_GROUP=%d" % g]) for g in range(INST_GROUPS)]
        else:
            jobs.append((s, s + ".o", []))
    return jobs


def _compile(src, name, extra):
    obj = os.path.join(BUILD, name)
    cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj, *extra]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("compile failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return obj, r.stderr


def build(force=False, verbose=False, ptxas_info=False):
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    info = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = _jobs()
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda j: _compile(j[0], j[1], j[2] + (info if j[0].endswith(".cu") else [])),
                              jobs))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
