"""3-D max pooling for GB300: Python binding of libmp3d.so.

The functions here carry the names of the C entry points declared in
``include/mp3d.h`` and only marshal arguments: they take CUDA tensors
(PyTorch is used for device memory and streams), pass raw device pointers,
sizes and the current stream to the library, and raise ``MP3DError`` on a
nonzero status. Every step of the computation runs in the library's CUDA
kernels; there is no CPU fallback. If the library has not been built, the
first call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmp3d.so")

F32, F16, BF16 = 0, 1, 2
BWD_AUTO, BWD_GATHER, BWD_ATOMIC = 0, 1, 2
DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

PATHS = {0: "noop", 1: "fwd_generic", 2: "fwd_s2", 3: "fwd_global", 4: "fwd_slab", 5: "fwd_padded",
         10: "bwd_disjoint",
         11: "bwd_overlap_tile", 12: "bwd_overlap_direct", 13: "bwd_atomic", 14: "bwd_overlap_roll",
         15: "bwd_padded", 19: "fwd_roll", 16: "bwd_recompute_k2s2", 17: "bwd_recompute_direct", 6: "fwd_ndhwc",
         18: "bwd_ndhwc"}

_lib = None


class MP3DError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({mp3d_status_string(status)})")


def lib() -> ctypes.CDLL:
    """The loaded libmp3d.so, with argument types set."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libmp3d.so not found at {LIB_PATH}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    pi32 = ctypes.POINTER(ctypes.c_int)
    L.maxpool3d_fwd.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 7 + [vp]
    L.adaptive_maxpool3d_fwd.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 4 + [vp]
    L.maxpool3d_bwd.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 11 + [vp, sz, vp]
    L.maxpool3d_bwd_workspace_bytes.argtypes = [i64] * 5 + [i32, i32]
    L.maxpool3d_bwd_workspace_bytes.restype = sz
    L.maxpool3d_fwd_plan.argtypes = [i64] * 5 + [i32] * 7 + [pi32]
    L.adaptive_maxpool3d_fwd_plan.argtypes = [i64] * 5 + [i32] * 4 + [pi32]
    L.maxpool3d_bwd_plan.argtypes = [i64] * 5 + [i32] * 11 + [pi32]
    L.maxpool3d_fwd_ex.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 14 + [vp]
    L.maxpool3d_bwd_ex.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 18 + [vp, sz, vp]
    L.maxpool3d_fwd_ex_plan.argtypes = [i64] * 5 + [i32] * 14 + [pi32]
    L.maxpool3d_bwd_ex_plan.argtypes = [i64] * 5 + [i32] * 18 + [pi32]
    L.maxpool3d_bwd_recompute.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 10 + [vp]
    L.maxpool3d_bwd_recompute_plan.argtypes = [i64] * 5 + [i32] * 10 + [pi32]
    L.maxpool3d_fwd_ndhwc.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 7 + [vp]
    L.adaptive_maxpool3d_fwd_ndhwc.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 4 + [vp]
    L.maxpool3d_bwd_ndhwc.argtypes = [vp, vp, vp] + [i64] * 5 + [i32] * 10 + [vp]
    L.mp3d_status_string.argtypes = [i32]
    L.mp3d_status_string.restype = ctypes.c_char_p
    for f in (L.maxpool3d_fwd, L.adaptive_maxpool3d_fwd, L.maxpool3d_bwd, L.maxpool3d_fwd_plan,
              L.adaptive_maxpool3d_fwd_plan, L.maxpool3d_bwd_plan, L.maxpool3d_fwd_ex,
              L.maxpool3d_bwd_ex, L.maxpool3d_fwd_ex_plan, L.maxpool3d_bwd_ex_plan,
              L.maxpool3d_bwd_recompute, L.maxpool3d_bwd_recompute_plan, L.maxpool3d_fwd_ndhwc,
              L.adaptive_maxpool3d_fwd_ndhwc, L.maxpool3d_bwd_ndhwc):
        f.restype = i32
    _lib = L
    return L


def mp3d_device_error_flags(clear: bool = True) -> int:
    """Device error flags (nonzero only if a kernel's bounded wait gave up)."""
    f = lib().mp3d_device_error_flags
    f.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
    f.restype = ctypes.c_int
    v = ctypes.c_uint(0)
    _check(f(ctypes.byref(v), 1 if clear else 0), "mp3d_device_error_flags")
    return v.value


def mp3d_status_string(status: int) -> str:
    return lib().mp3d_status_string(status).decode()


def _code(t: torch.Tensor) -> int:
    if t.dtype not in DTYPE_CODE:
        raise TypeError(f"unsupported dtype {t.dtype} (float32, float16, bfloat16 only)")
    return DTYPE_CODE[t.dtype]


def _cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError("tensors must be CUDA tensors (this library has no CPU path)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (NCDHW)")


def _ptr(t) -> int:
    """Device address of a tensor, or 0 (NULL) for None."""
    return 0 if t is None else t.data_ptr()


def _stream(t: torch.Tensor, stream):
    if stream is None:
        return torch.cuda.current_stream(t.device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str):
    if status != 0:
        raise MP3DError(status, where)


def pool_out_size(size, kernel, stride):
    """Output extent per axis for fixed windows without padding: (I - K) // S + 1."""
    return tuple((i - k) // s + 1 for i, k, s in zip(size, kernel, stride))


def pool_out_size_ex(size, kernel, stride, padding=(0, 0, 0), dilation=(1, 1, 1), ceil_mode=False):
    """Output extent per axis with padding, dilation and ceil mode (the rule
    documented for maxpool3d_fwd_ex); 0 where the arguments are invalid."""
    out = []
    for i, k, s, p, dl in zip(size, kernel, stride, padding, dilation):
        if i < 1 or k < 1 or s < 1 or dl < 1 or p < 0 or 2 * p > k:
            out.append(0)
            continue
        num = i + 2 * p - dl * (k - 1) - 1 + (s - 1 if ceil_mode else 0)
        o = num // s + 1
        if ceil_mode and (o - 1) * s >= i + p:
            o -= 1
        out.append(max(o, 0))
    return tuple(out)


def maxpool3d_fwd_ex(x, y, idx, kernel, stride, padding=(0, 0, 0), dilation=(1, 1, 1),
                     ceil_mode=False, stream=None):
    """Fixed-window forward with padding, dilation and ceil mode; idx None:
    values only."""
    _cuda(x, y, idx)
    N, C, D, H, W = x.shape
    with torch.cuda.device(x.device):
        st = lib().maxpool3d_fwd_ex(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W, *kernel,
                                    *stride, *padding, *dilation, int(bool(ceil_mode)), _code(x),
                                    _stream(x, stream))
    _check(st, "maxpool3d_fwd_ex")


def maxpool3d_bwd_ex(grad_out, idx, grad_in, kernel, stride, padding=(0, 0, 0), dilation=(1, 1, 1),
                     ceil_mode=False, algo=BWD_AUTO, workspace=None, stream=None):
    """Backward of maxpool3d_fwd_ex into caller-allocated grad_in."""
    _cuda(grad_out, idx, grad_in, workspace)
    N, C, D, H, W = grad_in.shape
    od, oh, ow = grad_out.shape[2:]
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd_ex(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(), N, C, D,
                                    H, W, od, oh, ow, *kernel, *stride, *padding, *dilation,
                                    int(bool(ceil_mode)), _code(grad_out), algo, ws, wsb,
                                    _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_ex")


def maxpool3d_fwd_ndhwc(x, y, idx, kernel, stride, stream=None):
    """Channels-last fixed-window forward: x (N, D, H, W, C), y and idx
    (N, OD, OH, OW, C); idx None: values only."""
    _cuda(x, y, idx)
    N, D, H, W, C = x.shape
    with torch.cuda.device(x.device):
        st = lib().maxpool3d_fwd_ndhwc(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W, *kernel,
                                       *stride, _code(x), _stream(x, stream))
    _check(st, "maxpool3d_fwd_ndhwc")


def adaptive_maxpool3d_fwd_ndhwc(x, y, idx, out_size, stream=None):
    """Channels-last adaptive-window forward."""
    _cuda(x, y, idx)
    N, D, H, W, C = x.shape
    with torch.cuda.device(x.device):
        st = lib().adaptive_maxpool3d_fwd_ndhwc(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W,
                                                *out_size, _code(x), _stream(x, stream))
    _check(st, "adaptive_maxpool3d_fwd_ndhwc")


def maxpool3d_bwd_ndhwc(grad_out, idx, grad_in, kernel=None, stride=None, stream=None):
    """Channels-last backward: grad_out and idx (N, OD, OH, OW, C), grad_in
    (N, D, H, W, C). kernel/stride None = adaptive windows."""
    _cuda(grad_out, idx, grad_in)
    N, D, H, W, C = grad_in.shape
    od, oh, ow = grad_out.shape[1:4]
    k = tuple(kernel) if kernel is not None else (0, 0, 0)
    s = tuple(stride) if stride is not None else (0, 0, 0)
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd_ndhwc(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(), N, C,
                                       D, H, W, od, oh, ow, *k, *s, _code(grad_out),
                                       _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_ndhwc")


def maxpool3d_bwd_recompute(x, grad_out, grad_in, kernel=None, stride=None, stream=None):
    """Backward without stored indices: the argmax of every window is
    recomputed from x. kernel/stride None = adaptive windows."""
    _cuda(x, grad_out, grad_in)
    N, C, D, H, W = grad_in.shape
    od, oh, ow = grad_out.shape[2:]
    k = tuple(kernel) if kernel is not None else (0, 0, 0)
    s = tuple(stride) if stride is not None else (0, 0, 0)
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd_recompute(x.data_ptr(), grad_out.data_ptr(), grad_in.data_ptr(), N,
                                           C, D, H, W, od, oh, ow, *k, *s, _code(grad_out),
                                           _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_recompute")


def maxpool3d_bwd_recompute_plan(in_shape, out_size, kernel, stride, dtype) -> str:
    p = ctypes.c_int(-1)
    k = tuple(kernel) if kernel is not None else (0, 0, 0)
    s = tuple(stride) if stride is not None else (0, 0, 0)
    _check(lib().maxpool3d_bwd_recompute_plan(*in_shape, *out_size, *k, *s, DTYPE_CODE[dtype],
                                              ctypes.byref(p)), "maxpool3d_bwd_recompute_plan")
    return PATHS[p.value]


def maxpool3d_fwd_ex_plan(in_shape, kernel, stride, padding, dilation, ceil_mode, dtype) -> str:
    p = ctypes.c_int(-1)
    _check(lib().maxpool3d_fwd_ex_plan(*in_shape, *kernel, *stride, *padding, *dilation,
                                       int(bool(ceil_mode)), DTYPE_CODE[dtype], ctypes.byref(p)),
           "maxpool3d_fwd_ex_plan")
    return PATHS[p.value]


def maxpool3d_bwd_ex_plan(in_shape, out_size, kernel, stride, padding, dilation, ceil_mode, dtype,
                          algo=BWD_AUTO) -> str:
    p = ctypes.c_int(-1)
    _check(lib().maxpool3d_bwd_ex_plan(*in_shape, *out_size, *kernel, *stride, *padding, *dilation,
                                       int(bool(ceil_mode)), DTYPE_CODE[dtype], algo, ctypes.byref(p)),
           "maxpool3d_bwd_ex_plan")
    return PATHS[p.value]


def maxpool3d_fwd(x, y, idx, kernel, stride, stream=None):
    """Fixed-window forward into caller-allocated y (x's dtype) and idx
    (int64); idx None: values only (no index is stored)."""
    _cuda(x, y, idx)
    N, C, D, H, W = x.shape
    with torch.cuda.device(x.device):
        st = lib().maxpool3d_fwd(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W,
                                 *kernel, *stride, _code(x), _stream(x, stream))
    _check(st, "maxpool3d_fwd")


def adaptive_maxpool3d_fwd(x, y, idx, out_size, stream=None):
    """Adaptive-window forward into caller-allocated y and idx; idx None:
    values only."""
    _cuda(x, y, idx)
    N, C, D, H, W = x.shape
    with torch.cuda.device(x.device):
        st = lib().adaptive_maxpool3d_fwd(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H,
                                          W, *out_size, _code(x), _stream(x, stream))
    _check(st, "adaptive_maxpool3d_fwd")


def maxpool3d_bwd_workspace_bytes(in_shape, dtype, algo=BWD_AUTO) -> int:
    N, C, D, H, W = in_shape
    return lib().maxpool3d_bwd_workspace_bytes(N, C, D, H, W, DTYPE_CODE[dtype], algo)


def maxpool3d_bwd(grad_out, idx, grad_in, kernel=None, stride=None, algo=BWD_AUTO,
                  workspace=None, stream=None):
    """Backward into caller-allocated grad_in. kernel/stride None = adaptive windows."""
    _cuda(grad_out, idx, grad_in, workspace)
    N, C, D, H, W = grad_in.shape
    od, oh, ow = grad_out.shape[2:]
    k = tuple(kernel) if kernel is not None else (0, 0, 0)
    s = tuple(stride) if stride is not None else (0, 0, 0)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(),
                                 N, C, D, H, W, od, oh, ow, *k, *s, _code(grad_out), algo,
                                 ws_ptr, ws_bytes, _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd")


def maxpool3d_fwd_plan(in_shape, kernel, stride, dtype) -> str:
    p = ctypes.c_int(-1)
    _check(lib().maxpool3d_fwd_plan(*in_shape, *kernel, *stride, DTYPE_CODE[dtype],
                                    ctypes.byref(p)), "maxpool3d_fwd_plan")
    return PATHS[p.value]


def adaptive_maxpool3d_fwd_plan(in_shape, out_size, dtype) -> str:
    p = ctypes.c_int(-1)
    _check(lib().adaptive_maxpool3d_fwd_plan(*in_shape, *out_size, DTYPE_CODE[dtype],
                                             ctypes.byref(p)), "adaptive_maxpool3d_fwd_plan")
    return PATHS[p.value]


def maxpool3d_bwd_plan(in_shape, out_size, kernel, stride, dtype, algo=BWD_AUTO) -> str:
    p = ctypes.c_int(-1)
    k = tuple(kernel) if kernel is not None else (0, 0, 0)
    s = tuple(stride) if stride is not None else (0, 0, 0)
    _check(lib().maxpool3d_bwd_plan(*in_shape, *out_size, *k, *s, DTYPE_CODE[dtype], algo,
                                    ctypes.byref(p)), "maxpool3d_bwd_plan")
    return PATHS[p.value]


def maxpool3d_bwd_noalloc(grad_out, idx, grad_in, kernel=None, stride=None, stream=None):
    """Atomic-form backward that allocates nothing: for callers that cannot
    allocate device memory while running. The binary32 accumulators (f16,
    bf16) live in a 32 MiB array inside the library, so N*C*D*H*W is limited
    to 8 Mi elements for those types; calls that overlap on the GPU race."""
    _cuda(grad_out, idx, grad_in)
    L = lib()
    f = L.maxpool3d_bwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 5 + [ctypes.c_int] * 10 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    N, C, D, H, W = grad_in.shape
    od, oh, ow = grad_out.shape[2:]
    k = tuple(kernel) if kernel is not None else (0, 0, 0)
    s = tuple(stride) if stride is not None else (0, 0, 0)
    with torch.cuda.device(grad_in.device):
        st = f(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(), N, C, D, H, W,
               od, oh, ow, *k, *s, _code(grad_out), _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_noalloc")
