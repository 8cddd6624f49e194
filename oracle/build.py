"""Compile the fp64 CPU oracle (``finalize_ref.c``) into a shared library.

TEST INFRASTRUCTURE ONLY: the library is loaded by the test suite, the smoke
check and the benchmark's CPU-baseline leg, never by the CUDA path.

Contraction of multiply-adds is switched off so that the oracle gives the
same doubles on x86-64 and on AArch64.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "finalize_ref.c")
SOURCES = [SRC, os.path.join(HERE, "routing_ref.c")]
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-shared", "-fPIC", "-Wall", "-Wextra"]


def compile_source(src_path, lib_path: str) -> str:
    """Compile C source(s) with the oracle's flags into ``lib_path``."""
    srcs = [src_path] if isinstance(src_path, str) else list(src_path)
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_FLAGS, "-o", tmp, *srcs, "-lm"], check=True)
    os.replace(tmp, lib_path)
    return lib_path


def build_oracle(force: bool = False) -> str:
    """Build ``_build/liboracle.so`` if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(LIB) >= os.path.getmtime(s) for s in SOURCES)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    return compile_source(SOURCES, LIB)


if __name__ == "__main__":
    print(build_oracle(force=True))
