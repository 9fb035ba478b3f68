"""CPU oracle for the NA3D forward pass (fp64, plain per-query loops in C).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The product path (the
CUDA library and its binding) never touches it, and it shares no code with
that path: the C source here has its own index arithmetic and bf16 widening.

The definition it follows is the one in "[Triton/Gluon] Add 3D neighborhood
flash attention (na3d_flash)" (ROCm/aiter pull request 5230): Motivation
(each token attends only to its KT x KH x KW neighbours) and Technical Details
(inward border shift, exactly KT*KH*KW keys per window, q pre-scaled by
head_dim^-0.5, exact per-query reference). See ``na3d_oracle.c`` for the
statement of the arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "na3d_oracle.c")
_LIB = os.path.join(_HERE, "libna3d_oracle.so")
_lib = None

_I64 = ctypes.c_int64
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the C oracle into ``libna3d_oracle.so`` (gcc, OpenMP)."""
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
        lib.na3d_oracle_window_start.argtypes = [_I64, _I64, _I64]
        lib.na3d_oracle_window_start.restype = _I64
        dims = [_I64] * 9
        lib.na3d_oracle_fwd.argtypes = [_P, _P, _P, _P] + dims + [ctypes.c_int]
        lib.na3d_oracle_fwd.restype = ctypes.c_int
        lib.na3d_oracle_fwd_rows.argtypes = [_P, _P, _P, _P, _I64, _P] + dims + [ctypes.c_int]
        lib.na3d_oracle_fwd_rows.restype = ctypes.c_int
        lib.na3d_oracle_row_detail.argtypes = [_P, _P, _P, _I64, _P, _P, _P] + dims
        lib.na3d_oracle_row_detail.restype = ctypes.c_int
        _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def _dims(q, kernel_size):
    if q.ndim != 6:
        raise ValueError("expected (B, T, H, W, NH, HD)")
    KT, KH, KW = (int(x) for x in kernel_size)
    return tuple(int(x) for x in q.shape) + (KT, KH, KW)


def window_start(i: int, K: int, N: int) -> int:
    """First key index of the window of query ``i`` on an axis of length N."""
    return int(_load().na3d_oracle_window_start(i, K, N))


def na3d_fwd(q, k, v, kernel_size, nthreads: int = 0) -> np.ndarray:
    """Full fp64 output (B,T,H,W,NH,HD) for bf16-bit inputs q, k, v."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v shapes differ")
    dims = _dims(q, kernel_size)
    out = np.empty(q.shape, dtype=np.float64)
    rc = _load().na3d_oracle_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                 out.ctypes.data, *dims, nthreads)
    if rc:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return out


def na3d_fwd_rows(q, k, v, kernel_size, rows, nthreads: int = 0) -> np.ndarray:
    """fp64 output rows for flat (b,t,h,w,n) indices ``rows``; shape (len(rows), HD)."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    dims = _dims(q, kernel_size)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, q.shape[-1]), dtype=np.float64)
    rc = _load().na3d_oracle_fwd_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                      rows.ctypes.data, rows.size, out.ctypes.data,
                                      *dims, nthreads)
    if rc:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return out


def na3d_row_detail(q, k, v, kernel_size, row: int):
    """(window token indices, softmax weights, output row) of one query row."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    dims = _dims(q, kernel_size)
    KK = dims[6] * dims[7] * dims[8]
    toks = np.empty(KK, dtype=np.int64)
    wts = np.empty(KK, dtype=np.float64)
    o = np.empty(q.shape[-1], dtype=np.float64)
    rc = _load().na3d_oracle_row_detail(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                        int(row), toks.ctypes.data, wts.ctypes.data,
                                        o.ctypes.data, *dims)
    if rc:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return toks, wts, o


# ---------------------------------------------------------------- QKV projection

def _widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def qkv_projection(x, w, bias, num_heads: int, head_dim: int) -> np.ndarray:
    """The fused QKV projection in fp64 (test infrastructure).

    x: bf16 bits (M, C); w: bf16 bits (3*NH*HD, C), q rows first, then k,
    then v; bias: bf16 bits (3*NH*HD,) or None. Returns fp64 (M, 3*NH*HD):
    x w^T + bias, with the q block (the first NH*HD columns) multiplied by
    head_dim^-0.5.

    The projection is the one the decoder attention uses: one concatenated
    Q/K/V weight whose output q, k, v are views of ("LTX-2.5 optimization:
    integrate faster AITER NA3D flash attention for diffusion decoder", xDiT
    pull request 773, Summary; Notes); the attention takes q pre-scaled by
    head_dim^-0.5 ("[Triton/Gluon] Add 3D neighborhood flash attention
    (na3d_flash)", Technical Details, launcher). A plain matrix product
    (library routine) on the exactly widened inputs; no blocking.
    """
    xf, wf = _widen_bf16(x), _widen_bf16(w)
    y = xf @ wf.T
    if bias is not None:
        y = y + _widen_bf16(bias)[None, :]
    nq = num_heads * head_dim
    y[:, :nq] *= head_dim ** -0.5
    return y
