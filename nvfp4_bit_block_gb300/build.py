"""Build the CUDA libraries in-tree with plain nvcc (one -gencode, sm_103a):

* nvfp4_bit_block_gb300/_build/libnvfp4.so -- the product library (the C ABI
  of include/nvfp4.h and its kernels);
* tests/selftest/_build/libnvfp4_selftest.so -- device self-checks used only
  by the tests (build_selftest); it holds no product entry point.

Translation units compile in parallel; the CUDA runtime is linked statically.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libnvfp4.so")
INCLUDE = os.path.join(ROOT, "include")
SELFTEST_DIR = os.path.join(ROOT, "tests", "selftest")
SELFTEST_BUILD = os.path.join(SELFTEST_DIR, "_build")
SELFTEST_LIB = os.path.join(SELFTEST_BUILD, "libnvfp4_selftest.so")

SOURCES = ["api.cu", "tmap.cu", "amax.cu", "quant1d.cu", "quant1d_sr.cu", "quant1d_46mae.cu", "quant1d_46mse.cu", "quant1d_46max.cu",
           "quant2d.cu", "dequant.cu", "analysis.cu", "gemm.cu"]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers():
    hs = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "nvfp4.h"))
    return hs


def _run(cmd, verbose=False):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(r.stdout, r.stderr)


def _build_lib(sources, build_dir, lib, force, verbose, extra_flags=()):
    """Compile `sources` (absolute paths) to objects in build_dir and link `lib`."""
    os.makedirs(build_dir, exist_ok=True)
    headers = _headers()
    nvcc = _nvcc()
    objs, jobs = [], []
    for s in sources:
        o = os.path.join(build_dir, os.path.basename(s).replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c", s, "-o", o])
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(lambda c: _run(c, verbose), jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        _run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "static", "-o", tmp, *objs],
             verbose)
        os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """The product library; returns its path."""
    return _build_lib([os.path.join(CSRC, s) for s in SOURCES], BUILD, LIB, force, verbose)


def build_selftest(force: bool = False, verbose: bool = False) -> str:
    """The test-only self-check library (its own copy of the tensor-map
    helper); returns its path."""
    srcs = [os.path.join(SELFTEST_DIR, "nvfp4_selftest.cu"), os.path.join(CSRC, "tmap.cu")]
    return _build_lib(srcs, SELFTEST_BUILD, SELFTEST_LIB, force, verbose)


if __name__ == "__main__":
    print(build(verbose=True))
    print(build_selftest(verbose=True))
