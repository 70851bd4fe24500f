"""Build the row-parallel CPU baseline (oracle/specdec_cpu_parallel.cpp) in-tree with g++.

Test and baseline infrastructure, like the oracle: tests/ and bench.py's CPU-baseline leg load
the library; the product path never does.  Rebuilt when the source or the flags change.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "specdec_cpu_parallel.cpp")
LIB = os.path.join(HERE, "libspecdec_cpu.so")
FLAGS = ["-O2", "-std=c++17", "-pthread", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("g++ not found: the CPU baseline cannot be built")
    h = hashlib.sha256()
    with open(SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(FLAGS).encode())
    h.update(os.uname().machine.encode())
    stamp = LIB + ".stamp"
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == h.hexdigest():
                return LIB
    tmp = LIB + ".tmp"
    r = subprocess.run([cxx] + FLAGS + [SRC, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"g++ failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(h.hexdigest())
    return LIB


def load():
    """The built library with its entry points' argument types set (ctypes)."""
    import ctypes
    lib = ctypes.CDLL(build())
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.cpu_verify_greedy.restype = i32
    lib.cpu_verify_greedy.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, i32]
    lib.cpu_verify_sample.restype = i32
    lib.cpu_verify_sample.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, ctypes.c_double, vp, vp,
                                      i32]
    lib.cpu_realign.restype = i32
    lib.cpu_realign.argtypes = ([vp, vp] + [i32] * 7 + [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                                         vp, ctypes.c_int32, i32])
    return lib


if __name__ == "__main__":
    print(build(force=True))
