"""Build libdr.so in-tree with nvcc for sm_103a.

``python -m recurrent_associative_memory_gb300.build`` (or ``build()``) compiles
every translation unit under csrc/ in parallel as relocatable device code and
links them into ``recurrent_associative_memory_gb300/libdr.so``.  No CMake, no
torch extension machinery: the library is plain CUDA C++ behind a C ABI.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdr.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-rdc=true", "-Xcompiler", "-fPIC",
         "-Xptxas", "-warn-spills", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdr")
    return path


def _run(cmd):
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + p.stdout + p.stderr)
    return p.stdout + p.stderr


def build(verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    cc = nvcc()
    cmds = [[cc, *ARCH, *FLAGS, *extra_flags, "-c", s, "-o", o] for s, o in zip(srcs, objs)]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(cmds))) as ex:
        logs = list(ex.map(_run, cmds))
    tmp = LIB + ".tmp"
    logs.append(_run([cc, *ARCH, "-rdc=true", "-shared", "-Xcompiler", "-fPIC", *objs,
                      "-o", tmp]))
    os.replace(tmp, LIB)
    if verbose:
        for s, log in zip(srcs + ["link"], logs):
            if log.strip():
                print(f"--- {os.path.basename(s)}\n{log}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
