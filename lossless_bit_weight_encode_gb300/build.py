"""Build libw12.so in-tree: the CUDA kernels for sm_103a (nvcc) plus the host
encoder and the C ABI (g++), linked with the static CUDA runtime so that the
library loads without a GPU driver present (only the calls need one)."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libw12.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CUDA_SOURCES = ["kernels.cu"]
CXX_SOURCES = ["encoder.cpp", "q8_host.cpp", "capi.cpp"]


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "w12.h"))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    jobs = []
    objs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        cmd = [NVCC, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xptxas", "-v", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj))
    for src in CXX_SOURCES:
        obj = os.path.join(OUT_DIR, src + ".o")
        cmd = [NVCC, "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-Wall,-Wextra,-pthread", "-I", INCLUDE,
               "-x", "cu" if src.endswith(".cu") else "c++", "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj))
    procs = [(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True), cmd, obj)
             for cmd, obj in jobs]
    for p, cmd, obj in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{out}")
        if verbose and out:
            sys.stdout.write(out)
        objs.append(obj)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-pthread", "-cudart", "static"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
