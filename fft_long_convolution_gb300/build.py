"""Compile the CUDA library (sm_103a) in-tree with nvcc."""
from __future__ import annotations

import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libfftconv_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
SOURCES = ["fftconv.cu", "mp_l16k.cu", "mp_l4k.cu", "mp_l16k_sparse.cu", "mp_l4k_sparse.cu", "mp_circ.cu"]  # compiled in parallel, then linked
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "fftconv.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libfftconv_gb300.so unless it is newer than every source."""
    with _lock:
        if not force and up_to_date():
            return LIB_PATH
        os.makedirs(BUILD_DIR, exist_ok=True)
        nvcc = os.environ.get("NVCC", "nvcc")
        tag = f".tmp{os.getpid()}"
        tmp = LIB_PATH + tag
        flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
        if verbose:
            flags.insert(0, "-Xptxas=-v")
        objs = [os.path.join(BUILD_DIR, os.path.splitext(s)[0] + tag + ".o") for s in SOURCES]

        def compile_one(i):
            subprocess.check_call([nvcc, *flags, "-c", "-o", objs[i], os.path.join(CSRC, SOURCES[i])])

        try:
            with ThreadPoolExecutor(len(SOURCES)) as ex:
                list(ex.map(compile_one, range(len(SOURCES))))
            subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
        finally:
            for o in objs:
                if os.path.exists(o):
                    os.remove(o)
        os.replace(tmp, LIB_PATH)
        return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
