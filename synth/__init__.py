"""Seeded synthetic inputs for the tests and the benchmark.

This module only produces input values; it holds none of the optimizer
step's arithmetic.  Both the CPU oracle (through ``host_fill`` /
``host_gather``) and the CUDA path (through ``dev_fill``, or a copy of a host
fill) take their inputs from here, and the two generators produce identical
bits (see ``gen.h`` for the definition: SplitMix64 words, Irwin-Hall(12)
approximate normal, one double multiply, round to fp32 / bf16).

Stream keys are derived from a seed and a tuple of small integers naming the
workload, the kind of tensor, the step, the rank and the micro-batch, so each
element of each input is addressable on its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
HOST_LIB = os.path.join(BUILD, "libsynth_host.so")
DEV_LIB = os.path.join(BUILD, "libsynth_dev.so")

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15

# tensor kinds used in stream keys
KIND_GRAD = 1
KIND_MASTER = 2
KIND_PARAM = 3
KIND_SHARD_BF16 = 4
KIND_OUTLIER = 5


def mix64(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, *fields: int) -> int:
    k = mix64(seed + GAMMA)
    for f in fields:
        k = mix64(k ^ mix64(int(f) + GAMMA))
    return k


class Stream(ctypes.Structure):
    _fields_ = [
        ("key", ctypes.c_uint64),
        ("key_out", ctypes.c_uint64),
        ("thr", ctypes.c_uint32),
        ("pad_", ctypes.c_uint32),
        ("sigma", ctypes.c_double),
        ("sigma_out", ctypes.c_double),
    ]

    def __repr__(self):
        return (f"Stream(key={self.key:#x}, thr={self.thr}, sigma={self.sigma}, "
                f"sigma_out={self.sigma_out})")


def normal_stream(seed: int, fields, sigma: float, outlier_p: float = 0.0,
                  outlier_scale: float = 100.0) -> Stream:
    """Approximately N(0, sigma) elements; with probability ``outlier_p`` an
    element is scaled by ``outlier_scale`` instead (selected per element by an
    independent key)."""
    fields = tuple(int(f) for f in fields)
    thr = int(round(outlier_p * (1 << 24)))
    return Stream(key=stream_key(seed, *fields),
                  key_out=stream_key(seed, *fields, KIND_OUTLIER) if thr else 0,
                  thr=thr, pad_=0, sigma=float(sigma),
                  sigma_out=float(sigma) * float(outlier_scale))


# ---------------------------------------------------------------- building

def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)


def build_host(force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(HERE, "synth_host.c")
    if force or not os.path.exists(HOST_LIB) or os.path.getmtime(HOST_LIB) < max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(HERE, "gen.h"))):
        tmp = HOST_LIB + f".tmp{os.getpid()}"
        _run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
              src, "-o", tmp])
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_dev(force: bool = False, arch: str = "103a") -> str:
    os.makedirs(BUILD, exist_ok=True)
    src = os.path.join(HERE, "synth_dev.cu")
    if force or not os.path.exists(DEV_LIB) or os.path.getmtime(DEV_LIB) < max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(HERE, "gen.h"))):
        tmp = DEV_LIB + f".tmp{os.getpid()}"
        _run(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC", "-fmad=false",
              f"-gencode=arch=compute_{arch},code=sm_{arch}", src, "-o", tmp])
        os.replace(tmp, DEV_LIB)
    return DEV_LIB


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        lib = ctypes.CDLL(build_host())
        P = ctypes.POINTER(Stream)
        lib.synth_fill_bf16.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.synth_fill_f32.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.synth_gather_bf16.argtypes = [P, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        lib.synth_gather_f32.argtypes = [P, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        lib.synth_fill_f16.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.synth_gather_f16.argtypes = [P, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        lib.synth_f32bits_to_f16.argtypes = [ctypes.c_uint32]
        lib.synth_f32bits_to_f16.restype = ctypes.c_uint16
        lib.synth_mix64.argtypes = [ctypes.c_uint64]
        lib.synth_mix64.restype = ctypes.c_uint64
        lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_normal.restype = ctypes.c_double
        lib.synth_is_outlier.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
        lib.synth_is_outlier.restype = ctypes.c_int
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            build_dev()
        lib = ctypes.CDLL(DEV_LIB)
        P = ctypes.POINTER(Stream)
        for name in ("synth_dev_fill_bf16", "synth_dev_fill_f32", "synth_dev_fill_f16"):
            f = getattr(lib, name)
            f.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            f.restype = ctypes.c_int
        _dev = lib
    return _dev


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# ---------------------------------------------------------------- host API

def host_fill(st: Stream, start: int, n: int, dtype: str, out: np.ndarray | None = None,
              nthreads: int | None = None) -> np.ndarray:
    """Elements start..start+n-1 as uint16 (bf16 / fp16 bits) or float32."""
    lib = _host_lib()
    if dtype == "f16":
        arr = out if out is not None else np.empty(n, dtype=np.uint16)
        assert arr.dtype == np.uint16 and arr.size == n and arr.flags.c_contiguous
        lib.synth_fill_f16(ctypes.byref(st), start, n, arr.ctypes.data, nthreads or _threads())
    elif dtype == "bf16":
        arr = out if out is not None else np.empty(n, dtype=np.uint16)
        assert arr.dtype == np.uint16 and arr.size == n and arr.flags.c_contiguous
        lib.synth_fill_bf16(ctypes.byref(st), start, n, arr.ctypes.data, nthreads or _threads())
    elif dtype == "f32":
        arr = out if out is not None else np.empty(n, dtype=np.float32)
        assert arr.dtype == np.float32 and arr.size == n and arr.flags.c_contiguous
        lib.synth_fill_f32(ctypes.byref(st), start, n, arr.ctypes.data, nthreads or _threads())
    else:
        raise ValueError(dtype)
    return arr


def host_gather(st: Stream, idx, dtype: str) -> np.ndarray:
    """Elements idx[i] (any order) as uint16 (bf16 bits) or float32."""
    lib = _host_lib()
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    if dtype == "f16":
        out = np.empty(idx.size, dtype=np.uint16)
        lib.synth_gather_f16(ctypes.byref(st), idx.ctypes.data, idx.size, out.ctypes.data)
    elif dtype == "bf16":
        out = np.empty(idx.size, dtype=np.uint16)
        lib.synth_gather_bf16(ctypes.byref(st), idx.ctypes.data, idx.size, out.ctypes.data)
    elif dtype == "f32":
        out = np.empty(idx.size, dtype=np.float32)
        lib.synth_gather_f32(ctypes.byref(st), idx.ctypes.data, idx.size, out.ctypes.data)
    else:
        raise ValueError(dtype)
    return out


def host_normal(key: int, n: int) -> float:
    return _host_lib().synth_normal(key, n)


# ---------------------------------------------------------------- device API

def dev_fill(st: Stream, tensor, start: int = 0) -> None:
    """Fill a contiguous CUDA tensor (torch.bfloat16, float16 or float32) with
    elements start..start+numel-1 of the stream, on torch's current stream."""
    import torch
    assert tensor.is_cuda and tensor.is_contiguous()
    lib = _dev_lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream(tensor.device).cuda_stream)
    if tensor.dtype == torch.bfloat16:
        rc = lib.synth_dev_fill_bf16(ctypes.byref(st), start, tensor.numel(),
                                     ctypes.c_void_p(tensor.data_ptr()), stream)
    elif tensor.dtype == torch.float16:
        rc = lib.synth_dev_fill_f16(ctypes.byref(st), start, tensor.numel(),
                                    ctypes.c_void_p(tensor.data_ptr()), stream)
    elif tensor.dtype == torch.float32:
        rc = lib.synth_dev_fill_f32(ctypes.byref(st), start, tensor.numel(),
                                    ctypes.c_void_p(tensor.data_ptr()), stream)
    else:
        raise TypeError(tensor.dtype)
    if rc != 0:
        raise RuntimeError("synthetic fill kernel failed to launch")


# ------------------------------------------------------- ranges of streams

def dev_fill_pieces(tensor, pieces, stream_of) -> None:
    """Fill ranges of a contiguous CUDA tensor from several streams:
    ``pieces`` lists (u, t, pos, start, count), and tensor[pos:pos + count]
    receives elements start..start+count-1 of ``stream_of(u, t)``.  Where the
    ranges come from (a FlatParameter layout) is the caller's business;
    positions no piece covers are left as they are."""
    for u, t, pos, start, count in pieces:
        if count:
            dev_fill(stream_of(u, t), tensor[pos:pos + count], start)


def host_gather_sources(units, tensors, index, stream_of, dtype: str) -> np.ndarray:
    """Element index[i] of ``stream_of(units[i], tensors[i])`` for every i, as
    uint16 (bf16 / fp16 bits) or float32; zero where tensors[i] < 0 (a
    position that holds no tensor element, e.g. padding)."""
    units = np.asarray(units, dtype=np.int64)
    tensors = np.asarray(tensors, dtype=np.int64)
    index = np.asarray(index, dtype=np.int64)
    out = np.zeros(index.size, dtype=np.float32 if dtype == "f32" else np.uint16)
    live = tensors >= 0
    if live.any():
        keys = np.unique(np.stack([units[live], tensors[live]], axis=1), axis=0)
        for u, t in keys:
            sel = np.nonzero(live & (units == u) & (tensors == t))[0]
            out[sel] = host_gather(stream_of(int(u), int(t)), index[sel], dtype)
    return out

