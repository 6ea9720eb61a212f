"""CPU oracle for 3-D max pooling (forward with argmax, backward routing).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline and reference legs of ``bench.py``. The product path
(``bwd_maxpool3d_fwd_gb300`` and its CUDA library) never imports it, and this
module imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, compiled with
gcc); this module only builds it and marshals torch CPU tensors into it.
Tensors are used as byte buffers: bfloat16 data is handed over as raw bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.c")
LIB = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle C source into a shared library (atomic replace)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, src, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.remove(tmp)
    return out


class Oracle:
    """One loaded build of the oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        P64 = ctypes.POINTER(i64)
        sig = {
            "oracle_f16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
            "oracle_bf16_to_f32": ([ctypes.c_uint16], ctypes.c_float),
            "oracle_f32_to_f16": ([ctypes.c_float], ctypes.c_uint16),
            "oracle_f32_to_bf16": ([ctypes.c_float], ctypes.c_uint16),
            "oracle_fixed_out_size": ([i64, i64, i64], i64),
            "oracle_fixed_window": ([i64, i64, i64, P64, P64], None),
            "oracle_adaptive_window": ([i64, i64, i64, P64, P64], None),
            "oracle_maxpool3d_fwd": ([i32, vp, vp, vp] + [i64] * 10, i32),
            "oracle_adaptive_maxpool3d_fwd": ([i32, vp, vp, vp] + [i64] * 7, i32),
            "oracle_maxpool3d_bwd": ([i32, vp, vp, vp, i64, i64, i64], i32),
            "oracle_ex_out_size": ([i64] * 5 + [i32], i64),
            "oracle_maxpool3d_fwd_ex": ([i32, vp, vp, vp] + [i64] * 16 + [i32], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        self.L = L
        self.path = path

    # ------------------------------------------------------------ scalars
    def f16_to_f32(self, bits: int) -> float:
        return self.L.oracle_f16_to_f32(bits)

    def bf16_to_f32(self, bits: int) -> float:
        return self.L.oracle_bf16_to_f32(bits)

    def f32_to_f16(self, v: float) -> int:
        return self.L.oracle_f32_to_f16(v)

    def f32_to_bf16(self, v: float) -> int:
        return self.L.oracle_f32_to_bf16(v)

    def fixed_out_size(self, I: int, K: int, S: int) -> int:
        """Output length along one axis for a fixed window, no padding (0 = invalid)."""
        return self.L.oracle_fixed_out_size(I, K, S)

    def fixed_window(self, o: int, K: int, S: int):
        s, e = ctypes.c_int64(), ctypes.c_int64()
        self.L.oracle_fixed_window(o, K, S, ctypes.byref(s), ctypes.byref(e))
        return s.value, e.value

    def adaptive_window(self, i: int, I: int, O: int):
        s, e = ctypes.c_int64(), ctypes.c_int64()
        self.L.oracle_adaptive_window(i, I, O, ctypes.byref(s), ctypes.byref(e))
        return s.value, e.value

    # ------------------------------------------------------------ tensors
    def maxpool3d_fwd(self, x: torch.Tensor, kernel, stride):
        """Fixed-window forward. x: (N, C, D, H, W) CPU tensor. Returns (y, idx)."""
        _check_cpu(x)
        N, C, D, H, W = x.shape
        kd, kh, kw = kernel
        sd, sh, sw = stride
        OD, OH, OW = (self.fixed_out_size(D, kd, sd), self.fixed_out_size(H, kh, sh),
                      self.fixed_out_size(W, kw, sw))
        if min(OD, OH, OW) < 1:
            raise ValueError("oracle: window does not fit the input")
        y = torch.empty((N, C, OD, OH, OW), dtype=x.dtype)
        idx = torch.empty((N, C, OD, OH, OW), dtype=torch.int64)
        rc = self.L.oracle_maxpool3d_fwd(_code(x), x.data_ptr(), y.data_ptr(), idx.data_ptr(),
                                         N * C, D, H, W, kd, kh, kw, sd, sh, sw)
        if rc:
            raise RuntimeError(f"oracle_maxpool3d_fwd failed ({rc})")
        return y, idx

    def adaptive_maxpool3d_fwd(self, x: torch.Tensor, out_size):
        """Adaptive-window forward. Returns (y, idx)."""
        _check_cpu(x)
        N, C, D, H, W = x.shape
        OD, OH, OW = out_size
        y = torch.empty((N, C, OD, OH, OW), dtype=x.dtype)
        idx = torch.empty((N, C, OD, OH, OW), dtype=torch.int64)
        rc = self.L.oracle_adaptive_maxpool3d_fwd(_code(x), x.data_ptr(), y.data_ptr(),
                                                  idx.data_ptr(), N * C, D, H, W, OD, OH, OW)
        if rc:
            raise RuntimeError(f"oracle_adaptive_maxpool3d_fwd failed ({rc})")
        return y, idx

    def ex_out_size(self, I: int, K: int, S: int, p: int, dl: int, ceil_mode: bool) -> int:
        """Output length with padding, dilation and ceil mode (0 = invalid)."""
        return self.L.oracle_ex_out_size(I, K, S, p, dl, 1 if ceil_mode else 0)

    def maxpool3d_fwd_ex(self, x: torch.Tensor, kernel, stride, padding, dilation, ceil_mode=False):
        """Forward with padding, dilation and ceil mode. Returns (y, idx)."""
        _check_cpu(x)
        N, C, D, H, W = x.shape
        out = tuple(self.ex_out_size(I, K, S, p, dl, ceil_mode)
                    for I, K, S, p, dl in zip((D, H, W), kernel, stride, padding, dilation))
        if min(out) < 1:
            raise ValueError("oracle: invalid window geometry")
        y = torch.empty((N, C) + out, dtype=x.dtype)
        idx = torch.empty((N, C) + out, dtype=torch.int64)
        rc = self.L.oracle_maxpool3d_fwd_ex(_code(x), x.data_ptr(), y.data_ptr(), idx.data_ptr(),
                                            N * C, D, H, W, *kernel, *stride, *padding, *dilation,
                                            1 if ceil_mode else 0)
        if rc:
            raise RuntimeError(f"oracle_maxpool3d_fwd_ex failed ({rc})")
        return y, idx

    def maxpool3d_bwd(self, grad_out: torch.Tensor, idx: torch.Tensor, in_spatial):
        """Route grad_out (N, C, OD, OH, OW) through idx into an (N, C, D, H, W) grad_in."""
        _check_cpu(grad_out, idx)
        if idx.dtype != torch.int64 or idx.shape != grad_out.shape:
            raise ValueError("oracle: idx must be int64 with grad_out's shape")
        N, C, OD, OH, OW = grad_out.shape
        D, H, W = in_spatial
        gin = torch.empty((N, C, D, H, W), dtype=grad_out.dtype)
        rc = self.L.oracle_maxpool3d_bwd(_code(grad_out), grad_out.data_ptr(), idx.data_ptr(),
                                         gin.data_ptr(), N * C, D * H * W, OD * OH * OW)
        if rc:
            raise RuntimeError(f"oracle_maxpool3d_bwd failed ({rc})")
        return gin


def _code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE_CODE:
        raise TypeError(f"oracle: unsupported dtype {t.dtype}")
    return _DTYPE_CODE[t.dtype]


def _check_cpu(*ts):
    for t in ts:
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("oracle: tensors must be contiguous CPU tensors")


_default = None


def default() -> Oracle:
    """The oracle built from oracle.c (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def __getattr__(name):
    # Module-level access to the default build: oracle.maxpool3d_fwd(...), etc.
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(default(), name)
