"""Build libmoe_finalize.so in-tree with nvcc for sm_103a.

The translation units are compiled in parallel and linked into one shared
library with the CUDA runtime linked statically, so the library loads
without any CUDA library path set up (it still needs the NVIDIA driver to
run kernels).
"""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_finalize.so")
SOURCES = ["finalize.cu", "allreduce.cu", "unfused.cu", "routing.cu", "api.cu", "noalloc.cu"]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3",
              "-std=c++17", "-Xcompiler", "-fPIC,-O2,-Wall", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "moe_finalize.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if needed) and return the path of libmoe_finalize.so.
    Concurrent builds (several processes finding the library out of date at
    once) are serialised by a lock file, so none of them reads another's
    half-written objects."""
    if not force and not _stale():
        build_fastcall()
        return LIB
    import fcntl
    os.makedirs(OBJ_DIR, exist_ok=True)
    with open(os.path.join(OBJ_DIR, "build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and not _stale():      # another process built it meanwhile
            build_fastcall()
            return LIB
        return _build_locked(verbose, extra_flags)


def _build_locked(verbose, extra_flags) -> str:
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-cudart", "static", "-gencode", "arch=compute_103a,code=sm_103a",
           "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    build_fastcall()
    return LIB


FASTCALL_SRC = os.path.join(CSRC, "fastcall.c")


def build_fastcall() -> str:
    """Compile the _fastcall CPython extension (direct and bound calls of
    moe_finalize_ex; no CUDA code) next to the library; returns its path, or
    "" when the Python headers are not available (the binding then uses
    ctypes for every call)."""
    import sysconfig
    inc = sysconfig.get_paths()["include"]
    out = os.path.join(PKG, "_fastcall" + sysconfig.get_config_var("EXT_SUFFIX"))
    if not os.path.exists(os.path.join(inc, "Python.h")):
        return ""
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(FASTCALL_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    r = subprocess.run(["gcc", "-O2", "-shared", "-fPIC", "-Wall", "-I", inc, "-o", tmp,
                        FASTCALL_SRC], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"gcc failed on fastcall.c:\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build_library(force=True, verbose=True, extra_flags=sys.argv[1:]))
