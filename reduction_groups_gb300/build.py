"""Build the in-tree native libraries (no cmake, no pip install).

* ``_build/libpsk.so``          the C-ABI library: CUDA kernels for sm_103a plus
                                host validation, cudart linked statically;
* ``_build/libpsk_hostmath.so`` the device exp/erf source compiled as plain C++
                                for the host, used only by tests that check the
                                device math element by element on the CPU.

Every translation unit compiles in parallel; arithmetic flags keep IEEE
semantics (no fused multiply-add contraction, IEEE division and square root,
no flush to zero), because results must be bit-identical to the unfused chain.
"""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

CU_SOURCES = ["group.cu", "softmax.cu", "adamw.cu"]
CPP_SOURCES = ["api.cpp"]

NVCC_FLAGS = [
    ARCH, "-O3", "-lineinfo", "-std=c++17",
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC,-ffp-contract=off",
    "--threads", "2",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    """Compile both libraries if any source changed; returns the libpsk path."""
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".inc", ".h"))]
    headers.append(os.path.join(HERE, "..", "include", "psk.h"))
    jobs = []
    objs = []
    for src in CU_SOURCES + CPP_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers):
            flags = list(NVCC_FLAGS)
            if ptxas_info and src.endswith(".cu"):
                flags += ["-Xptxas", "-v"]
            jobs.append([nvcc, *flags, "-c", s, "-o", o])
    hostmath = os.path.join(OUT, "libpsk_hostmath.so")
    hm_src = os.path.join(CSRC, "crmath_host.cpp")
    cxx = shutil.which("g++") or "g++"
    if force or _stale(hostmath, [hm_src] + headers):
        jobs.append([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                     hm_src, "-o", hostmath])
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        outs = list(ex.map(_run, jobs))
    if verbose:
        for o in outs:
            if o.strip():
                print(o)
    lib = os.path.join(OUT, "libpsk.so")
    if force or jobs or not os.path.exists(lib):
        _run([nvcc, ARCH, "-shared", "-o", lib, *objs, "-cudart", "static"])
    return lib


if __name__ == "__main__":
    import sys

    print(build(verbose=True, force="--force" in sys.argv, ptxas_info="--ptxas" in sys.argv))
