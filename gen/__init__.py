"""Seeded synthetic inputs shared by the GPU path and the oracle.

Thin ctypes wrapper over ``gen/philox_gen.cpp`` (Philox4x32-10 counter-based
streams, Box-Muller normals, multiply-shift targets).  It holds none of the
loss arithmetic.  Every function can produce any contiguous slice of a tensor
(``offset`` in elements) so that a few rows of a multi-GB tensor can be made on
the host without making the rest.

Stream ids used for the workloads: 0 = logits or student input, 1 = targets,
2 = (student) head weight, 3 = teacher input, 4 = teacher head weight.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "philox_gen.cpp")
LIB = os.path.join(HERE, "_build", "libgen.so")

STREAM_LOGITS = 0
STREAM_X = 0
STREAM_TARGET = 1
STREAM_W = 2
STREAM_XT = 3
STREAM_WT = 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator library with g++ (portable flags only)."""
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread",
                               SRC, "-o", tmp])
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            u64, u32, i64, dbl, vp, ci = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64,
                                          ctypes.c_double, ctypes.c_void_p, ctypes.c_int)
            lib.gen_philox4x32_10.argtypes = [vp, vp, vp]
            for name in ("gen_normal_f64", "gen_normal_f32", "gen_normal_bf16"):
                getattr(lib, name).argtypes = [u64, u32, u64, u64, dbl, vp, ci]
            lib.gen_targets.argtypes = [u64, u32, u64, u64, i64, vp, ci]
            _lib = lib
    return _lib


def _threads(threads):
    return int(threads) if threads else (os.cpu_count() or 1)


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().gen_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def _dst(shape, dtype, out):
    n = int(np.prod(shape)) if len(shape) else 1
    if out is None:
        arr = np.empty(shape, dtype=dtype)
        return arr, arr.ctypes.data, n
    # torch tensor or numpy array supplied by the caller (must be contiguous, host)
    if hasattr(out, "data_ptr"):
        assert out.is_contiguous() and out.device.type == "cpu" and out.numel() == n
        return out, out.data_ptr(), n
    assert out.flags.c_contiguous and out.size == n
    return out, out.ctypes.data, n


def normal_f64(seed, stream, shape, sigma=1.0, offset=0, out=None, threads=None):
    arr, ptr, n = _dst(shape, np.float64, out)
    _load().gen_normal_f64(seed, stream, offset, n, float(sigma), ptr, _threads(threads))
    return arr


def normal_f32(seed, stream, shape, sigma=1.0, offset=0, out=None, threads=None):
    arr, ptr, n = _dst(shape, np.float32, out)
    _load().gen_normal_f32(seed, stream, offset, n, float(sigma), ptr, _threads(threads))
    return arr


def normal_bf16_bits(seed, stream, shape, sigma=1.0, offset=0, out=None, threads=None):
    """bf16 values as their uint16 bit patterns (numpy has no bf16)."""
    arr, ptr, n = _dst(shape, np.uint16, out)
    _load().gen_normal_bf16(seed, stream, offset, n, float(sigma), ptr, _threads(threads))
    return arr


def targets(seed, stream, shape, V, offset=0, out=None, threads=None):
    arr, ptr, n = _dst(shape, np.int64, out)
    _load().gen_targets(seed, stream, offset, n, int(V), ptr, _threads(threads))
    return arr


def bf16_bits_to_f32(bits):
    """Exact widening of bf16 bit patterns to float32 (numpy)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)
