"""Python binding of the GB300 NA3D forward library (``libna3d.so``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/na3d.h``. There is no CPU or
PyTorch fallback; if the library has not been built, importing works but any
call raises ``NA3DUnavailable``.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "NA3DError", "NA3DUnavailable", "na3d_attention", "na3d_fwd", "na3d_fwd_strided", "na3d_fwd_region",
    "na3d_qkv_proj", "qkv_views", "na3d_status_string", "na3d_plan",
    "na3d_device_status", "library_path", "load_library", "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libna3d.so")
EXPORTED_SYMBOLS = ("na3d_fwd", "na3d_fwd_strided", "na3d_fwd_region", "na3d_qkv_proj",
                    "na3d_selftest_withhold", "na3d_status_string", "na3d_plan",
                    "na3d_device_status")

NA3D_OK = 0
_I64 = ctypes.c_int64
_P = ctypes.c_void_p
_lib = None


class NA3DError(RuntimeError):
    """A non-zero status returned by the C ABI."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {na3d_status_string(status)} (status {status})")


class NA3DUnavailable(RuntimeError):
    """The CUDA library is missing: build it with ``__graft_entry__.build()``."""


class PlanInfo(ctypes.Structure):
    _fields_ = [("bt", ctypes.c_int32), ("bh", ctypes.c_int32), ("bw", ctypes.c_int32),
                ("cw", ctypes.c_int32), ("cr", ctypes.c_int32), ("n_mma", ctypes.c_int32),
                ("hd_box", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("bricks_per_slice", ctypes.c_int64), ("chunks_per_slice", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int64), ("w_stride", ctypes.c_int32),
                ("tile_cap", ctypes.c_int32)]


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load ``libna3d.so`` (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise NA3DUnavailable(
            f"{LIB_PATH} is missing; build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    lib.na3d_fwd.argtypes = [_P, _P, _P, _P] + [_I64] * 9 + [_P]
    lib.na3d_fwd.restype = ctypes.c_int
    lib.na3d_fwd_strided.argtypes = [_P, _P, _P, _P] + [_I64] * 12 + [_P]
    lib.na3d_fwd_strided.restype = ctypes.c_int
    lib.na3d_fwd_region.argtypes = [_P, _P, _P, _P] + [_I64] * 18 + [_P]
    lib.na3d_fwd_region.restype = ctypes.c_int
    lib.na3d_qkv_proj.argtypes = [_P, _P, _P, _P] + [_I64] * 4 + [_P]
    lib.na3d_qkv_proj.restype = ctypes.c_int
    lib.na3d_selftest_withhold.argtypes = [_P, _P, _P, _P] + [_I64] * 10 + [_P]
    lib.na3d_selftest_withhold.restype = ctypes.c_int
    lib.na3d_status_string.argtypes = [ctypes.c_int]
    lib.na3d_status_string.restype = ctypes.c_char_p
    lib.na3d_plan.argtypes = [_I64] * 8 + [ctypes.POINTER(PlanInfo)]
    lib.na3d_plan.restype = ctypes.c_int
    lib.na3d_device_status.argtypes = [_P]
    lib.na3d_device_status.restype = ctypes.c_int
    _lib = lib
    return lib


def na3d_status_string(status: int) -> str:
    return load_library().na3d_status_string(int(status)).decode()


_torch = None
_cuda_ok = None   # torch.cuda.is_available(), fixed for the process


def _torch_module():
    global _torch, _cuda_ok
    if _torch is None:
        import torch
        _torch = torch
        _cuda_ok = torch.cuda.is_available()
    return _torch


def _check_bf16_on_device(tensors):
    """Each (name, tensor) is a bf16 tensor on the current CUDA device: the
    kernels get raw pointers, so a host or other-device tensor must not pass."""
    torch = _torch_module()
    dev = torch.cuda.current_device() if _cuda_ok else -2
    for name, t in tensors:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype is not torch.bfloat16 or t.get_device() != dev:
            raise TypeError(f"{name} must be a bfloat16 tensor on the current CUDA device")


def _stream_handle(stream) -> int:
    if stream is None:   # the current torch stream of the current device
        torch = _torch_module()
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def na3d_fwd(q, k, v, out, kernel_size, stream=None) -> None:
    """out = NA3D(q, k, v) for bf16 CUDA tensors of shape (B, T, H, W, NH, HD).

    ``q`` must already be scaled by HD**-0.5. ``kernel_size`` = (KT, KH, KW),
    odd. ``out`` is written in place. Runs asynchronously on ``stream``
    (default: the current torch stream). Raises NA3DError on a bad argument.
    """
    lib = _lib if _lib is not None else load_library()
    _check_bf16_on_device((("q", q), ("k", k), ("v", v), ("out", out)))
    shape = q.shape
    if len(shape) != 6 or k.shape != shape or v.shape != shape or out.shape != shape:
        raise ValueError("q, k, v and out must have the same 6-D (B,T,H,W,NH,HD) shape")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous() and out.is_contiguous()):
        raise ValueError("q, k, v and out must be contiguous")
    KT, KH, KW = (int(x) for x in kernel_size)
    rc = lib.na3d_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                      *shape, KT, KH, KW, _stream_handle(stream))
    if rc != NA3D_OK:
        raise NA3DError(rc, "na3d_fwd")


def na3d_attention(q, k, v, kernel_size, stream=None):
    """Returns a new tensor out = NA3D(q, k, v): ``na3d_fwd`` with the output
    allocated like ``q`` (contiguous bf16 (B, T, H, W, NH, HD) on its device).
    q must already be scaled by HD**-0.5."""
    torch = _torch_module()
    out = torch.empty_like(q, memory_format=torch.contiguous_format)
    na3d_fwd(q, k, v, out, kernel_size, stream=stream)
    return out


def _token_stride(name, t) -> int:
    """Elements between consecutive (b,t,h,w) positions of a (B,T,H,W,NH,HD)
    view whose heads are packed (head stride HD, unit element stride)."""
    st, sh = t.stride(), t.shape
    if st[5] != 1 or (sh[4] > 1 and st[4] != sh[5]):
        raise ValueError(f"{name}: heads must be packed (strides [..., HD, 1])")
    for i in (2, 1, 0):
        if sh[i] > 1 and st[i] != sh[i + 1] * st[i + 1]:
            raise ValueError(f"{name}: grid positions must share one token stride")
    return int(st[3])


def na3d_fwd_strided(q, k, v, out, kernel_size, stream=None) -> None:
    """``na3d_fwd`` for q, k, v views with a token stride, e.g. the three
    slices ``x[..., 0, :, :]``, ``x[..., 1, :, :]``, ``x[..., 2, :, :]`` of a
    fused projection output ``x`` of shape (B, T, H, W, 3, NH, HD). ``out`` is
    a contiguous (B, T, H, W, NH, HD) bf16 CUDA tensor."""
    lib = load_library()
    _check_bf16_on_device((("q", q), ("k", k), ("v", v), ("out", out)))
    for t in (q, k, v, out):
        if t.dim() != 6 or tuple(t.shape) != tuple(q.shape):
            raise ValueError("q, k, v and out must have the same 6-D shape")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    strides = [_token_stride(n, t) for n, t in (("q", q), ("k", k), ("v", v))]
    KT, KH, KW = (int(x) for x in kernel_size)
    rc = lib.na3d_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              *[int(x) for x in q.shape], KT, KH, KW, *strides,
                              _stream_handle(stream))
    if rc != NA3D_OK:
        raise NA3DError(rc, "na3d_fwd_strided")


def na3d_fwd_region(q, k, v, out, kernel_size, offset, stream=None) -> None:
    """``out`` = the rows of NA3D on the whole grid at the query box
    ``offset`` = (t0, h0, w0) with the extents of ``q``: q and out have shape
    (B, Tq, Hq, Wq, NH, HD), k and v (B, T, H, W, NH, HD). Every query keeps
    its window in the whole grid (global coordinates). q, k, v may be views
    with a token stride as in ``na3d_fwd_strided``; ``out`` is contiguous."""
    lib = load_library()
    _check_bf16_on_device((("q", q), ("k", k), ("v", v), ("out", out)))
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dim() != 6:
            raise ValueError(f"{name} must be a 6-D tensor")
    if tuple(k.shape) != tuple(v.shape) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("k and v must share a shape, and so must q and out")
    if q.shape[0] != k.shape[0] or q.shape[4:] != k.shape[4:]:
        raise ValueError("q and k must agree on B, NH and HD")
    if not out.is_contiguous():
        raise ValueError("out must be contiguous")
    strides = [_token_stride(n, t) for n, t in (("q", q), ("k", k), ("v", v))]
    KT, KH, KW = (int(x) for x in kernel_size)
    t0, h0, w0 = (int(x) for x in offset)
    B, T, H, W, NH, HD = (int(x) for x in k.shape)
    Tq, Hq, Wq = (int(x) for x in q.shape[1:4])
    rc = lib.na3d_fwd_region(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             B, T, H, W, NH, HD, KT, KH, KW, t0, h0, w0, Tq, Hq, Wq,
                             *strides, _stream_handle(stream))
    if rc != NA3D_OK:
        raise NA3DError(rc, "na3d_fwd_region")


def na3d_qkv_proj(x, w, bias, qkv, num_heads, head_dim, stream=None) -> None:
    """qkv = x w^T (+ bias), the q block scaled by head_dim**-0.5 (see
    ``na3d_qkv_proj`` in include/na3d.h). x: contiguous bf16 CUDA tensor
    (..., C); w: (3*NH*HD, C); bias: (3*NH*HD,) or None; qkv: contiguous bf16
    with x's leading dimensions and 3*NH*HD elements per token, e.g.
    (B, T, H, W, 3, NH, HD). ``qkv_views`` gives the attention inputs."""
    lib = load_library()
    tensors = [("x", x), ("w", w), ("qkv", qkv)] + ([("bias", bias)] if bias is not None else [])
    _check_bf16_on_device(tensors)
    for name, t in tensors:
        if not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    NH, HD = int(num_heads), int(head_dim)
    C = int(x.shape[-1])
    M = x.numel() // C if C else 0
    N = 3 * NH * HD
    if tuple(w.shape) != (N, C) or (bias is not None and tuple(bias.shape) != (N,)):
        raise ValueError("w must be (3*NH*HD, C) and bias (3*NH*HD,)")
    if qkv.numel() != M * N:
        raise ValueError("qkv must hold 3*NH*HD values per token of x")
    rc = lib.na3d_qkv_proj(x.data_ptr(), w.data_ptr(), bias.data_ptr() if bias is not None else None,
                           qkv.data_ptr(), M, C, NH, HD, _stream_handle(stream))
    if rc != NA3D_OK:
        raise NA3DError(rc, "na3d_qkv_proj")


def qkv_views(qkv):
    """q, k, v views (B, T, H, W, NH, HD) of a (B, T, H, W, 3, NH, HD)
    projection output, for ``na3d_fwd_strided``."""
    return qkv[..., 0, :, :], qkv[..., 1, :, :], qkv[..., 2, :, :]


def na3d_plan(T, H, W, NH, HD, KT, KH, KW) -> dict:
    """The tiling ``na3d_fwd`` uses for this problem (host only, no GPU)."""
    info = PlanInfo()
    rc = load_library().na3d_plan(T, H, W, NH, HD, KT, KH, KW, ctypes.byref(info))
    if rc != NA3D_OK:
        raise NA3DError(rc, "na3d_plan")
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_}


def na3d_device_status(stream=None) -> int:
    """Synchronize ``stream``; NA3D_ERR_DEVICE_TIMEOUT if a kernel wait gave up."""
    return int(load_library().na3d_device_status(_stream_handle(stream)))
