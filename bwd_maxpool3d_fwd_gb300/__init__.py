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
         18: "bwd_ndhwc", 20: "bwd_ndhwc_roll"}

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
    L.maxpool3d_bwd_ndhwc_plan.argtypes = [i64] * 5 + [i32] * 10 + [pi32]
    L.maxpool3d_out_size.argtypes = [i64] * 3 + [i32] * 6 + [pi32] * 3
    L.maxpool3d_ex_out_size.argtypes = [i64] * 3 + [i32] * 13 + [pi32] * 3
    L.mp3d_status_string.argtypes = [i32]
    L.mp3d_status_string.restype = ctypes.c_char_p
    for f in (L.maxpool3d_fwd, L.adaptive_maxpool3d_fwd, L.maxpool3d_bwd, L.maxpool3d_fwd_plan,
              L.adaptive_maxpool3d_fwd_plan, L.maxpool3d_bwd_plan, L.maxpool3d_fwd_ex,
              L.maxpool3d_bwd_ex, L.maxpool3d_fwd_ex_plan, L.maxpool3d_bwd_ex_plan,
              L.maxpool3d_bwd_recompute, L.maxpool3d_bwd_recompute_plan, L.maxpool3d_fwd_ndhwc,
              L.adaptive_maxpool3d_fwd_ndhwc, L.maxpool3d_bwd_ndhwc, L.maxpool3d_bwd_ndhwc_plan,
              L.maxpool3d_out_size,
              L.maxpool3d_ex_out_size):
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
    dev = None
    for t in ts:
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError("tensors must be CUDA tensors (this library has no CPU path)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on different devices ({dev} and {t.device})")


def _dims5(t, what):
    if t.dim() != 5:
        raise ValueError(f"{what} must be 5-D, got shape {tuple(t.shape)}")
    return tuple(int(v) for v in t.shape)


def _expect(t, shape, dtype, what):
    """A caller buffer must have exactly the shape and type the call writes or reads."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{what}: dtype {t.dtype}, expected {dtype}")


def _window_args(kernel, stride):
    k = tuple(kernel) if kernel is not None else (0, 0, 0)
    s = tuple(stride) if stride is not None else (0, 0, 0)
    return k, s


def _bwd_out(grad_out, grad_in, kernel, stride, channels_last=False):
    """Check a backward call's buffers against the sizes the library computes.
    Returns (N, C, D, H, W) and the output size (od, oh, ow)."""
    gi = _dims5(grad_in, "grad_in")
    go = _dims5(grad_out, "grad_out")
    if channels_last:
        N, D, H, W, C = gi
        out = go[1:4]
        want = (N,) + out + (C,)
    else:
        N, C, D, H, W = gi
        out = go[2:]
        want = (N, C) + out
    if kernel is not None or stride is not None:
        k, s = _window_args(kernel, stride)
        fixed = pool_out_size((D, H, W), k, s)
        if tuple(out) != fixed:
            raise ValueError(f"grad_out spatial size {tuple(out)}, the window gives {fixed}")
    _expect(grad_out, want, grad_in.dtype, "grad_out")
    return (N, C, D, H, W), tuple(out)


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
    """Output extent (OD, OH, OW) of the fixed-window forward without padding,
    from the library (maxpool3d_out_size); raises MP3DError when the library
    rejects the input size or the window."""
    od, oh, ow = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().maxpool3d_out_size(*size, *kernel, *stride, ctypes.byref(od), ctypes.byref(oh),
                                    ctypes.byref(ow)), "maxpool3d_out_size")
    return (od.value, oh.value, ow.value)


def pool_out_size_ex(size, kernel, stride, padding=(0, 0, 0), dilation=(1, 1, 1), ceil_mode=False):
    """Output extent with padding, dilation and ceil mode, from the library
    (maxpool3d_ex_out_size); raises MP3DError when the geometry is rejected."""
    od, oh, ow = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().maxpool3d_ex_out_size(*size, *kernel, *stride, *padding, *dilation,
                                       int(bool(ceil_mode)), ctypes.byref(od), ctypes.byref(oh),
                                       ctypes.byref(ow)), "maxpool3d_ex_out_size")
    return (od.value, oh.value, ow.value)


def maxpool3d_fwd(x, y, idx, kernel, stride, stream=None):
    """Fixed-window forward into caller-allocated y (x's dtype) and idx
    (int64), both shaped (N, C) + pool_out_size(...); idx None: values only
    (no index is stored)."""
    N, C, D, H, W = _dims5(x, "x")
    out = (N, C) + pool_out_size((D, H, W), kernel, stride)
    _expect(y, out, x.dtype, "y")
    _expect(idx, out, torch.int64, "idx")
    _cuda(x, y, idx)
    with torch.cuda.device(x.device):
        st = lib().maxpool3d_fwd(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W,
                                 *kernel, *stride, _code(x), _stream(x, stream))
    _check(st, "maxpool3d_fwd")


def adaptive_maxpool3d_fwd(x, y, idx, out_size, stream=None):
    """Adaptive-window forward into caller-allocated y and idx, shaped
    (N, C) + out_size; idx None: values only."""
    N, C, D, H, W = _dims5(x, "x")
    out = (N, C) + tuple(int(v) for v in out_size)
    _expect(y, out, x.dtype, "y")
    _expect(idx, out, torch.int64, "idx")
    _cuda(x, y, idx)
    with torch.cuda.device(x.device):
        st = lib().adaptive_maxpool3d_fwd(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H,
                                          W, *out_size, _code(x), _stream(x, stream))
    _check(st, "adaptive_maxpool3d_fwd")


def maxpool3d_bwd_workspace_bytes(in_shape, dtype, algo=BWD_AUTO) -> int:
    N, C, D, H, W = in_shape
    return lib().maxpool3d_bwd_workspace_bytes(N, C, D, H, W, DTYPE_CODE[dtype], algo)


def _workspace(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def maxpool3d_bwd(grad_out, idx, grad_in, kernel=None, stride=None, algo=BWD_AUTO,
                  workspace=None, stream=None):
    """Backward into caller-allocated grad_in. grad_out and idx (int64) are
    shaped (N, C, od, oh, ow), grad_in (N, C, D, H, W) of grad_out's type.
    kernel/stride None = adaptive windows."""
    (N, C, D, H, W), (od, oh, ow) = _bwd_out(grad_out, grad_in, kernel, stride)
    _expect(idx, grad_out.shape, torch.int64, "idx")
    k, s = _window_args(kernel, stride)
    ws_ptr, ws_bytes = _workspace(workspace)
    _cuda(grad_out, idx, grad_in, workspace)
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(),
                                 N, C, D, H, W, od, oh, ow, *k, *s, _code(grad_out), algo,
                                 ws_ptr, ws_bytes, _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd")


def maxpool3d_fwd_ex(x, y, idx, kernel, stride, padding=(0, 0, 0), dilation=(1, 1, 1),
                     ceil_mode=False, stream=None):
    """Fixed-window forward with padding, dilation and ceil mode; y and idx
    shaped (N, C) + pool_out_size_ex(...); idx None: values only."""
    N, C, D, H, W = _dims5(x, "x")
    out = (N, C) + pool_out_size_ex((D, H, W), kernel, stride, padding, dilation, ceil_mode)
    _expect(y, out, x.dtype, "y")
    _expect(idx, out, torch.int64, "idx")
    _cuda(x, y, idx)
    with torch.cuda.device(x.device):
        st = lib().maxpool3d_fwd_ex(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W, *kernel,
                                    *stride, *padding, *dilation, int(bool(ceil_mode)), _code(x),
                                    _stream(x, stream))
    _check(st, "maxpool3d_fwd_ex")


def maxpool3d_bwd_ex(grad_out, idx, grad_in, kernel, stride, padding=(0, 0, 0), dilation=(1, 1, 1),
                     ceil_mode=False, algo=BWD_AUTO, workspace=None, stream=None):
    """Backward of maxpool3d_fwd_ex into caller-allocated grad_in."""
    N, C, D, H, W = _dims5(grad_in, "grad_in")
    _dims5(grad_out, "grad_out")
    od, oh, ow = pool_out_size_ex((D, H, W), kernel, stride, padding, dilation, ceil_mode)
    _expect(grad_out, (N, C, od, oh, ow), grad_in.dtype, "grad_out")
    _expect(idx, (N, C, od, oh, ow), torch.int64, "idx")
    ws, wsb = _workspace(workspace)
    _cuda(grad_out, idx, grad_in, workspace)
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd_ex(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(), N, C, D,
                                    H, W, od, oh, ow, *kernel, *stride, *padding, *dilation,
                                    int(bool(ceil_mode)), _code(grad_out), algo, ws, wsb,
                                    _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_ex")


def maxpool3d_fwd_ndhwc(x, y, idx, kernel, stride, stream=None):
    """Channels-last fixed-window forward: x (N, D, H, W, C), y and idx
    (N, OD, OH, OW, C); idx None: values only."""
    N, D, H, W, C = _dims5(x, "x")
    out = (N,) + pool_out_size((D, H, W), kernel, stride) + (C,)
    _expect(y, out, x.dtype, "y")
    _expect(idx, out, torch.int64, "idx")
    _cuda(x, y, idx)
    with torch.cuda.device(x.device):
        st = lib().maxpool3d_fwd_ndhwc(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W, *kernel,
                                       *stride, _code(x), _stream(x, stream))
    _check(st, "maxpool3d_fwd_ndhwc")


def adaptive_maxpool3d_fwd_ndhwc(x, y, idx, out_size, stream=None):
    """Channels-last adaptive-window forward."""
    N, D, H, W, C = _dims5(x, "x")
    out = (N,) + tuple(int(v) for v in out_size) + (C,)
    _expect(y, out, x.dtype, "y")
    _expect(idx, out, torch.int64, "idx")
    _cuda(x, y, idx)
    with torch.cuda.device(x.device):
        st = lib().adaptive_maxpool3d_fwd_ndhwc(x.data_ptr(), y.data_ptr(), _ptr(idx), N, C, D, H, W,
                                                *out_size, _code(x), _stream(x, stream))
    _check(st, "adaptive_maxpool3d_fwd_ndhwc")


def maxpool3d_bwd_ndhwc(grad_out, idx, grad_in, kernel=None, stride=None, stream=None):
    """Channels-last backward: grad_out and idx (N, OD, OH, OW, C), grad_in
    (N, D, H, W, C). kernel/stride None = adaptive windows."""
    (N, C, D, H, W), (od, oh, ow) = _bwd_out(grad_out, grad_in, kernel, stride, channels_last=True)
    _expect(idx, grad_out.shape, torch.int64, "idx")
    k, s = _window_args(kernel, stride)
    _cuda(grad_out, idx, grad_in)
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd_ndhwc(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(), N, C,
                                       D, H, W, od, oh, ow, *k, *s, _code(grad_out),
                                       _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_ndhwc")


def maxpool3d_bwd_recompute(x, grad_out, grad_in, kernel=None, stride=None, stream=None):
    """Backward without stored indices: the argmax of every window is
    recomputed from x (shaped and typed like grad_in). kernel/stride None =
    adaptive windows."""
    (N, C, D, H, W), (od, oh, ow) = _bwd_out(grad_out, grad_in, kernel, stride)
    _expect(x, grad_in.shape, grad_in.dtype, "x")
    k, s = _window_args(kernel, stride)
    _cuda(x, grad_out, grad_in)
    with torch.cuda.device(grad_in.device):
        st = lib().maxpool3d_bwd_recompute(x.data_ptr(), grad_out.data_ptr(), grad_in.data_ptr(), N,
                                           C, D, H, W, od, oh, ow, *k, *s, _code(grad_out),
                                           _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_recompute")


def maxpool3d_bwd_noalloc(grad_out, idx, grad_in, kernel=None, stride=None, stream=None):
    """Atomic-form backward that allocates nothing: for callers that cannot
    allocate device memory while running. The binary32 accumulators (f16,
    bf16) live in a 32 MiB array inside the library, so N*C*D*H*W is limited
    to 8 Mi elements for those types; calls that overlap on the GPU race."""
    (N, C, D, H, W), (od, oh, ow) = _bwd_out(grad_out, grad_in, kernel, stride)
    _expect(idx, grad_out.shape, torch.int64, "idx")
    L = lib()
    f = L.maxpool3d_bwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 5 + [ctypes.c_int] * 10 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    k, s = _window_args(kernel, stride)
    _cuda(grad_out, idx, grad_in)
    with torch.cuda.device(grad_in.device):
        st = f(grad_out.data_ptr(), idx.data_ptr(), grad_in.data_ptr(), N, C, D, H, W,
               od, oh, ow, *k, *s, _code(grad_out), _stream(grad_in, stream))
    _check(st, "maxpool3d_bwd_noalloc")


# ------------------------------------------------------------ plan queries

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
    k, s = _window_args(kernel, stride)
    _check(lib().maxpool3d_bwd_plan(*in_shape, *out_size, *k, *s, DTYPE_CODE[dtype], algo,
                                    ctypes.byref(p)), "maxpool3d_bwd_plan")
    return PATHS[p.value]


def maxpool3d_bwd_ndhwc_plan(in_shape, out_size, kernel, stride, dtype) -> str:
    """Kernel of maxpool3d_bwd_ndhwc for 16-byte aligned buffers; in_shape is
    (N, C, D, H, W) whatever the layout. kernel/stride None = adaptive."""
    p = ctypes.c_int(-1)
    k, s = _window_args(kernel, stride)
    _check(lib().maxpool3d_bwd_ndhwc_plan(*in_shape, *out_size, *k, *s, DTYPE_CODE[dtype],
                                          ctypes.byref(p)), "maxpool3d_bwd_ndhwc_plan")
    return PATHS[p.value]


def maxpool3d_bwd_recompute_plan(in_shape, out_size, kernel, stride, dtype) -> str:
    p = ctypes.c_int(-1)
    k, s = _window_args(kernel, stride)
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
