"""Seeded synthetic NA3D inputs (q, k, v) as bf16 bit patterns.

Random numbers only: this module holds none of the attention arithmetic, so
both the CPU oracle and the CUDA path may consume what it generates.

Recipe (the workload of the NA3D forward kernel on its benchmark shapes):
q, k, v are iid N(0,1), contiguous (B, T, H, W, NH, HD), drawn from one
splitmix64 stream in the order q, then k, then v, each in layout order; q is
multiplied by fp32(HD**-0.5) in fp32 before its single rounding to bf16,
because the operation takes q already scaled by head_dim**-0.5.

The generator itself is C (``gen.c``), compiled on first use with gcc.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libna3d_inputs.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``libna3d_inputs.so`` next to it (atomic rename)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.na3d_gen_normal_bf16.argtypes = [
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_float,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
        lib.na3d_gen_normal_bf16.restype = None
        lib.na3d_gen_normal_f64.argtypes = [
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
        lib.na3d_gen_normal_f64.restype = None
        _lib = lib
    return _lib


def q_scale(hd: int) -> float:
    """fp32 value of HD**-0.5 (computed in fp64, rounded once to fp32)."""
    return float(np.float32(1.0 / math.sqrt(hd)))


def fill_bf16(ptr: int, n: int, seed: int, counter_base: int,
              scale: float | None = None, nthreads: int = 0) -> None:
    """Write n bf16 normals z[counter_base + i] (times fp32 ``scale``) to ``ptr``.

    ``ptr`` is a host address (numpy buffer or pinned torch tensor)."""
    _load().na3d_gen_normal_bf16(
        ctypes.c_uint64(seed), ctypes.c_uint64(counter_base), ctypes.c_int64(n),
        ctypes.c_float(scale if scale is not None else 1.0),
        1 if scale is not None else 0, ctypes.c_void_p(ptr), nthreads)


def normals_f64(n: int, seed: int = 0, counter_base: int = 0) -> np.ndarray:
    """fp64 normals before any rounding (for tests of the generator)."""
    out = np.empty(n, dtype=np.float64)
    _load().na3d_gen_normal_f64(ctypes.c_uint64(seed), ctypes.c_uint64(counter_base),
                                ctypes.c_int64(n), out.ctypes.data)
    return out


def fill_qkv_host(q_ptr: int, k_ptr: int, v_ptr: int, shape, seed: int = 0,
                  nthreads: int = 0) -> None:
    """Fill three host buffers of ``shape`` = (B,T,H,W,NH,HD) with the recipe."""
    n = int(np.prod(shape))
    hd = int(shape[-1])
    fill_bf16(q_ptr, n, seed, 0, q_scale(hd), nthreads)
    fill_bf16(k_ptr, n, seed, n, None, nthreads)
    fill_bf16(v_ptr, n, seed, 2 * n, None, nthreads)


def make_qkv(B: int, T: int, H: int, W: int, NH: int, HD: int, seed: int = 0,
             nthreads: int = 0):
    """Return q, k, v as uint16 arrays (bf16 bit patterns) of shape (B,T,H,W,NH,HD)."""
    shape = (B, T, H, W, NH, HD)
    q = np.empty(shape, dtype=np.uint16)
    k = np.empty(shape, dtype=np.uint16)
    v = np.empty(shape, dtype=np.uint16)
    fill_qkv_host(q.ctypes.data, k.ctypes.data, v.ctypes.data, shape, seed, nthreads)
    return q, k, v


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (via fp32, nearest even)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)
