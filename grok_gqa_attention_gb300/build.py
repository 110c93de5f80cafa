"""Build libgrok_attn.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each .cu file is compiled in parallel, then linked into one shared library
next to this file. The CUDA runtime is linked statically; the driver's
tensor-map encoder is looked up at run time, so no libcuda link is needed.
"""
from __future__ import annotations

import concurrent.futures
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build", platform.machine())
LIB = os.path.join(PKG, "libgrok_attn.so")
SOURCES = ["abi.cu", "rope_append.cu", "prefill.cu", "decode.cu", "selftest.cu", "pipe.cu", "qkv.cu", "slots.cu", "int8_small.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _stamp_path() -> str:
    return os.path.join(BUILD, "lib.stamp")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "grok_attn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(_stamp_path())):
        return False
    with open(_stamp_path()) as f:
        if f.read().strip() != platform.machine():
            return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *CFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = "".join(msg for _, msg in results)
    if verbose or ptxas_info:
        print(log)
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(_stamp_path(), "w") as f:
        f.write(platform.machine())
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write(log)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))
