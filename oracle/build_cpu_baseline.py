"""Compile the benchmark's CPU baseline loop (cpu_decode_fp32.c) into a shared library.

Test and benchmark infrastructure, like the rest of oracle/: gcc -O2 with OpenMP
(without it when the compiler has no OpenMP runtime, then the loop runs on one core).
The build is skipped when the library is newer than the source.  Returns the library
path, or None when no C compiler is available."""

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cpu_decode_fp32.c")
LIB = os.path.join(HERE, "_build", "libcpu_decode_fp32.so")


def build():
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        return None
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + ".tmp"
    base = [cc, "-O2", "-std=c11", "-shared", "-fPIC", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"CPU baseline build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def load():
    """The compiled loop as a ctypes function (building it first), or None."""
    import ctypes
    path = build()
    if path is None:
        return None
    f = ctypes.CDLL(path).tq_cpu_decode_turbo4
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp,
                  ctypes.c_float, vp, ctypes.c_int]
    return f
