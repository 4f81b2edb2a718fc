"""Builds libsvp.so in place: nvcc for sm_103a, one object per translation
unit compiled in parallel, then one shared-library link.  No cmake."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsvp.so")
SOURCES = ["attention.cu", "attention_tc.cu", "accept.cu", "kv_append.cu",
           "api.cu", "noalloc.cu", "step.cu"]
HEADERS = [os.path.join(CSRC, h)
           for h in ("ptx.cuh", "svp_internal.h", "attn_common.cuh")] + [
    os.path.join(INCLUDE, "svp.h")]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", INCLUDE, "-I", CSRC]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC] + FLAGS + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link libsvp.so (in place)."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, defines, force: bool = False) -> str:
    """A separately named copy of the library (libsvp_<name>.so beside
    libsvp.so) compiled with extra preprocessor definitions, e.g. the test
    build whose producers stall so that the bounded waits run out."""
    lib = os.path.join(PKG, f"libsvp_{name}.so")
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS
    if (not force and os.path.exists(lib) and
            all(os.path.getmtime(d) <= os.path.getmtime(lib) for d in deps)):
        return lib
    out_dir = os.path.join(BUILD_DIR, name)
    os.makedirs(out_dir, exist_ok=True)
    extra = [f"-D{d}" for d in defines]

    def one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [NVCC] + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([NVCC] + ARCH + ["-shared", "-o", tmp] + objs,
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv)
    print(LIB)
