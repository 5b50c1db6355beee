"""Builds libshardstep.so in-tree for sm_103a with nvcc (no torch extension
machinery, no cmake).  The translation units are compiled in parallel and
linked into sharded_optimizer_step_gb300/libshardstep.so."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libshardstep.so")

SOURCES = ["step.cu", "step_tma.cu", "copy.cu", "accum_step.cu", "fsdp2_step.cu", "state.cu",
           "api.cpp", "ckpt.cpp", "ready.cpp"]
HEADERS = ["common.cuh", "internal.h"]
ARCH = "103a"


def nvcc_flags(arch: str = ARCH, ptxas_verbose: bool = False):
    flags = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo", "-fmad=false",
             f"-gencode=arch=compute_{arch},code=sm_{arch}", "-I", INCLUDE, "-I", CSRC]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    return flags


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, arch: str = ARCH, verbose: bool = False) -> str:
    """Compile and link the library if any source is newer than it."""
    os.makedirs(OBJ, exist_ok=True)
    deps_common = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "shardstep.h")]
    procs, objs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + deps_common):
            cmd = ["nvcc", *nvcc_flags(arch, verbose), "-c", s, "-o", o]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("nvcc failed: " + " ".join(cmd) + "\n" + out)
        if verbose and out:
            print(out, file=sys.stderr)
    if force or procs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["nvcc", "-shared", f"-gencode=arch=compute_{arch},code=sm_{arch}", *objs, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
