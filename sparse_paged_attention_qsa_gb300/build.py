"""Build libqsa.so in-tree for sm_103a with nvcc (no cmake, no torch).

    python -m sparse_paged_attention_qsa_gb300.build [--force] [--ptxas-info]

Each .cu under csrc/ compiles to an object in parallel; the objects link
into ``sparse_paged_attention_qsa_gb300/libqsa.so`` (cudart linked
statically).  Objects go to ``_build/`` next to this file.

``build_wait_test()`` builds ``libqsa_waittest.so``, a test-only variant of
the selection and attention entry points compiled with QSA_WAIT_TEST: its
stage waits give up after 2 ms and it exports one extra symbol that makes
the first CTA of the score kernel (or of the fused small-batch kernel) leave
one stage fill without a copy, so the failure-detection test can make a
device wait run out.  The product library
carries neither.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqsa.so")
WAIT_TEST_LIB = os.path.join(PKG, "libqsa_waittest.so")
WAIT_TEST_SOURCES = ("qsa_abi.cu", "qsa_select.cu", "qsa_attention.cu", "qsa_fused.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqsa")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + \
        [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _build_lib(lib: str, srcs, objdir: str, defines=(), ptxas_info: bool = False,
               verbose: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)
    inc = ["-I", INCLUDE, "-I", CSRC]
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + [f"-D{d}" for d in defines]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, *inc, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp,
           *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, ptxas_info: bool = False, verbose: bool = False) -> str:
    if not force and not ptxas_info and up_to_date():
        return LIB
    return _build_lib(LIB, _sources(), BUILD, ptxas_info=ptxas_info, verbose=verbose)


def build_wait_test(force: bool = False) -> str:
    """The test-only variant (see the module docstring)."""
    if not force and up_to_date(WAIT_TEST_LIB):
        return WAIT_TEST_LIB
    srcs = [os.path.join(CSRC, n) for n in WAIT_TEST_SOURCES]
    return _build_lib(WAIT_TEST_LIB, srcs, os.path.join(BUILD, "waittest"),
                      defines=("QSA_WAIT_TEST",))


if __name__ == "__main__":
    build(force="--force" in sys.argv, ptxas_info="--ptxas-info" in sys.argv,
          verbose="-v" in sys.argv)
    print(LIB)
