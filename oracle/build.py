"""Compiles the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, no CUDA.  Host-portable flags only (the same source builds on the
x86-64 development host and the aarch64 GPU hosts).  ``real="f32"`` builds the
float instantiation of the same source (oracle/liboracle_f32.so), which only the
benchmark's CPU-baseline leg times; parity always uses the double build.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
LIB_F32 = os.path.join(HERE, "liboracle_f32.so")


def build(force: bool = False, real: str = "f64") -> str:
    lib = LIB if real == "f64" else LIB_F32
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(SRC):
        return lib
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           *([] if real == "f64" else ["-DORACLE_REAL=float"]), "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
    print(build(force="--force" in sys.argv, real="f32"))
