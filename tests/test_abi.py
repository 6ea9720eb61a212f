"""The C ABI without a GPU: the library builds and loads, exports every
function the header declares, rejects bad arguments before any CUDA call,
and plans the expected kernel path for each workload."""
import ctypes
import os
import re

import pytest
import torch

import bwd_maxpool3d_fwd_gb300 as mp
from bwd_maxpool3d_fwd_gb300 import build as mp_build
from bwd_maxpool3d_fwd_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, NULLPTR, SHAPE, WINDOW, DTYPE, WORKSPACE, CUDA, ALGO, ALIGN, ALIAS = range(10)


@pytest.fixture(scope="module")
def L():
    mp_build.build()
    return mp.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "mp3d.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^(?:int|size_t|const char\*)\s+(\w+)\s*\(", src, flags=re.M)


def test_header_symbols_exported(L):
    names = header_functions()
    assert {"maxpool3d_fwd", "adaptive_maxpool3d_fwd", "maxpool3d_bwd"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in mp3d.h but not exported"


def test_status_strings(L):
    for s in range(10):
        assert mp.mp3d_status_string(s)
    assert mp.mp3d_status_string(99) == "unknown status"


# Host buffers are enough: every call below fails validation before any
# CUDA call, so no pointer is ever dereferenced.
@pytest.fixture(scope="module")
def bufs():
    a = (ctypes.c_char * 4096)()
    b = (ctypes.c_char * 4096)()
    c = (ctypes.c_char * 4096)()
    return ctypes.addressof(a), ctypes.addressof(b), ctypes.addressof(c), (a, b, c)


def fwd(L, x, y, i, N=1, C=1, D=4, H=4, W=4, k=(2, 2, 2), s=(2, 2, 2), dt=0):
    return L.maxpool3d_fwd(x, y, i, N, C, D, H, W, *k, *s, dt, None)


def test_fwd_argument_errors(L, bufs):
    x, y, i, _ = bufs
    assert fwd(L, None, y, i) == NULLPTR
    assert fwd(L, x, None, i) == NULLPTR
    # idx NULL asks for the values-only forward: the other checks still apply
    # (each case below fails before any CUDA call)
    assert fwd(L, x, y, None, dt=3) == DTYPE
    assert fwd(L, x + 1, y, None, dt=1) == ALIGN
    assert fwd(L, x, x + 64, None) == ALIAS
    assert fwd(L, x, None, None) == NULLPTR
    assert fwd(L, x, y, i, D=0) == SHAPE
    assert fwd(L, x, y, i, N=-1) == SHAPE
    assert fwd(L, x, y, i, k=(0, 2, 2)) == WINDOW
    assert fwd(L, x, y, i, s=(2, 0, 2)) == WINDOW
    assert fwd(L, x, y, i, k=(5, 2, 2)) == WINDOW
    assert fwd(L, x, y, i, dt=3) == DTYPE
    assert fwd(L, x + 1, y, i, dt=1) == ALIGN
    assert fwd(L, x, y, i + 4) == ALIGN
    assert fwd(L, x, x + 64, i) == ALIAS
    assert fwd(L, x, y, y + 8) == ALIAS
    big = 1 << 11
    assert fwd(L, x, y, i, D=big, H=big, W=big) == SHAPE          # plane volume >= 2^31
    # empty input: a no-op (no CUDA call), even with NULL pointers
    assert fwd(L, None, None, None, N=0) == OK
    assert fwd(L, None, None, None, C=0, k=(0, 1, 1)) == WINDOW   # still validated


def test_adaptive_argument_errors(L, bufs):
    x, y, i, _ = bufs
    f = L.adaptive_maxpool3d_fwd
    assert f(x, y, i, 1, 1, 4, 4, 4, 0, 2, 2, 0, None) == SHAPE
    assert f(x, y, i, 1, 1, 4, 4, 4, 2, 2, 2, 5, None) == DTYPE
    assert f(None, y, i, 1, 1, 4, 4, 4, 2, 2, 2, 0, None) == NULLPTR
    assert f(None, None, None, 0, 3, 4, 4, 4, 9, 9, 9, 0, None) == OK   # O > I accepted


def bwd(L, g, i, gi, od=(2, 2, 2), k=(2, 2, 2), s=(2, 2, 2), dt=0, algo=0, ws=None, wsb=0,
        D=4, H=4, W=4, N=1, C=1):
    return L.maxpool3d_bwd(g, i, gi, N, C, D, H, W, *od, *k, *s, dt, algo, ws, wsb, None)


def test_bwd_argument_errors(L, bufs):
    g, i, gi, _ = bufs
    assert bwd(L, None, i, gi) == NULLPTR
    assert bwd(L, g, i, gi, od=(3, 2, 2)) == WINDOW         # sizes must match the window
    assert bwd(L, g, i, gi, k=(2, 0, 2)) == WINDOW           # partly adaptive
    assert bwd(L, g, i, gi, od=(0, 2, 2), k=(0, 0, 0), s=(0, 0, 0)) == SHAPE
    assert bwd(L, g, i, gi, algo=3) == ALGO
    assert bwd(L, g, i, gi, dt=9) == DTYPE
    assert bwd(L, g, i, gi, dt=1, algo=2) == WORKSPACE       # f16 atomic needs binary32 room
    assert bwd(L, g, i, gi, dt=1, algo=2, ws=g + 2048, wsb=64) == WORKSPACE
    assert bwd(L, g, i, g + 16) == ALIAS


def test_workspace_bytes(L):
    n = 2 * 3 * 4 * 5 * 6
    assert L.maxpool3d_bwd_workspace_bytes(2, 3, 4, 5, 6, 1, 2) == 4 * n
    assert L.maxpool3d_bwd_workspace_bytes(2, 3, 4, 5, 6, 2, 2) == 4 * n
    assert L.maxpool3d_bwd_workspace_bytes(2, 3, 4, 5, 6, 0, 2) == 0
    assert L.maxpool3d_bwd_workspace_bytes(2, 3, 4, 5, 6, 1, 0) == 0
    assert L.maxpool3d_bwd_workspace_bytes(2, 3, 0, 5, 6, 1, 2) == 0


def test_stated_output_sizes():
    for w in workloads.WORKLOADS:
        if w.mode == "fixed":
            assert mp.pool_out_size((w.D, w.H, w.W), w.kernel, w.stride) == tuple(w.out)


def test_plans_per_workload(L):
    expect_fwd = {0: {"fwd_slab"}, 1: {"fwd_roll"}, 2: {"fwd_s2"}, 3: {"fwd_s2"},
                  4: {"fwd_global"}}
    expect_bwd = {0: {"bwd_disjoint"}, 1: {"bwd_overlap_roll"}, 2: {"bwd_disjoint"},
                  3: {"bwd_overlap_roll"}, 4: {"bwd_disjoint"}}
    for n, w in enumerate(workloads.WORKLOADS):
        if w.mode == "fixed":
            pf = mp.maxpool3d_fwd_plan(w.in_shape, w.kernel, w.stride, w.dtype)
            pb = mp.maxpool3d_bwd_plan(w.in_shape, w.out, w.kernel, w.stride, w.dtype)
        else:
            pf = mp.adaptive_maxpool3d_fwd_plan(w.in_shape, w.out, w.dtype)
            pb = mp.maxpool3d_bwd_plan(w.in_shape, w.out, None, None, w.dtype)
        assert pf in expect_fwd[n], (w.name, pf)
        assert pb in expect_bwd[n], (w.name, pb)
        pa = mp.maxpool3d_bwd_plan(w.in_shape, w.out, w.kernel if w.mode == "fixed" else None,
                                   w.stride if w.mode == "fixed" else None, w.dtype,
                                   mp.BWD_ATOMIC)
        assert pa == "bwd_atomic"


def test_channels_last_backward_plans(L):
    # the rolling scatter for overlapping or adaptive windows when 16 bytes
    # of channels divide C; the gather for windows that tile the input, odd
    # channel counts, and windows with three covers per axis
    f16, bf16, f32 = torch.float16, torch.bfloat16, torch.float32
    plan = mp.maxpool3d_bwd_ndhwc_plan
    for dt in (f16, bf16, f32):
        assert plan((32, 128, 16, 112, 112), (7, 55, 55), (3, 3, 3), (2, 2, 2), dt) == "bwd_ndhwc_roll"
        assert plan((8, 64, 32, 64, 64), (16, 32, 32), (2, 2, 2), (2, 2, 2), dt) == "bwd_ndhwc"
        assert plan((2, 16, 10, 30, 29), (4, 11, 10), None, None, dt) == "bwd_ndhwc_roll"
        assert plan((2, 5, 7, 9, 10), (6, 4, 3), (2, 3, 2), (1, 2, 3), dt) == "bwd_ndhwc"   # odd C
        assert plan((1, 8, 9, 9, 9), (3, 3, 3), (5, 5, 5), (2, 2, 2), dt) == "bwd_ndhwc"    # 3 covers
    assert plan((1, 12, 8, 17, 35), (3, 8, 17), (3, 3, 3), (2, 2, 2), f32) == "bwd_ndhwc_roll"
    assert plan((1, 12, 8, 17, 35), (3, 8, 17), (3, 3, 3), (2, 2, 2), f16) == "bwd_ndhwc"
    assert plan((0, 16, 8, 17, 35), (3, 8, 17), (3, 3, 3), (2, 2, 2), f16) == "noop"


def test_plan_rules(L):
    # fixed kernel == input on every axis: a global reduction
    assert mp.maxpool3d_fwd_plan((2, 2, 3, 4, 5), (3, 4, 5), (1, 1, 1), torch.float32) == "fwd_global"
    # kernel <= stride everywhere: disjoint, including gaps (kernel < stride)
    assert mp.maxpool3d_bwd_plan((1, 1, 9, 9, 9), (3, 3, 3), (2, 2, 2), (3, 3, 3),
                                 torch.float16) == "bwd_disjoint"
    # adaptive output larger than the input: overlapping
    assert mp.maxpool3d_bwd_plan((1, 1, 3, 3, 3), (5, 5, 5), None, None,
                                 torch.float32) != "bwd_disjoint"
    assert mp.maxpool3d_fwd_plan((0, 4, 3, 3, 3), (2, 2, 2), (1, 1, 1), torch.float32) == "noop"
    # at most two windows over any position on every axis: the rolling scatter
    assert mp.maxpool3d_bwd_plan((1, 1, 9, 9, 9), (4, 4, 4), (3, 3, 3), (2, 2, 2),
                                 torch.bfloat16) == "bwd_overlap_roll"
    assert mp.maxpool3d_bwd_plan((1, 1, 9, 9, 9), (8, 8, 8), (2, 2, 2), (1, 1, 1),
                                 torch.float32) == "bwd_overlap_roll"
    # three windows over a position along d only: the tiled owner gather
    assert mp.maxpool3d_bwd_plan((1, 1, 9, 8, 8), (7, 4, 4), (3, 2, 2), (1, 2, 2),
                                 torch.float16) == "bwd_overlap_tile"
    # three windows over a position on every axis (kernel 3, stride 1; adaptive
    # 3 -> 5 has windows [0,1) [0,2) [1,2) [1,3) [2,3)): the direct gather
    assert mp.maxpool3d_bwd_plan((1, 1, 9, 9, 9), (7, 7, 7), (3, 3, 3), (1, 1, 1),
                                 torch.float16) == "bwd_overlap_direct"
    assert mp.maxpool3d_bwd_plan((1, 1, 3, 3, 3), (5, 5, 5), None, None,
                                 torch.float32) == "bwd_overlap_direct"


def test_binding_rejects_cpu_tensors(L):
    x = torch.zeros((1, 1, 4, 4, 4))
    with pytest.raises(ValueError):
        mp.maxpool3d_fwd(x, x, x, (2, 2, 2), (2, 2, 2))


def fwd_ex(L, x, y, i, N=1, C=1, D=6, H=6, W=6, k=(3, 3, 3), s=(2, 2, 2), p=(1, 1, 1), dl=(1, 1, 1),
           cm=0, dt=0):
    return L.maxpool3d_fwd_ex(x, y, i, N, C, D, H, W, *k, *s, *p, *dl, cm, dt, None)


def test_padded_argument_errors(L, bufs):
    # every case fails validation before any CUDA call (host buffers)
    x, y, i, _ = bufs
    assert fwd_ex(L, x, y, i, p=(2, 1, 1)) == WINDOW             # padding above half the kernel
    assert fwd_ex(L, x, y, i, p=(-1, 0, 0)) == WINDOW
    assert fwd_ex(L, x, y, i, dl=(0, 1, 1)) == WINDOW
    assert fwd_ex(L, x, y, i, cm=2) == WINDOW
    assert fwd_ex(L, x, y, i, D=1, k=(4, 3, 3), p=(0, 1, 1)) == WINDOW    # no output
    # dilation 3 with padding 1 on a length-1 axis: the window {-1, 2} holds no input
    assert fwd_ex(L, x, y, i, D=1, k=(2, 3, 3), s=(1, 2, 2), p=(1, 1, 1), dl=(3, 1, 1)) == WINDOW
    assert fwd_ex(L, x, y, i, dt=3) == DTYPE
    assert fwd_ex(L, None, y, i) == NULLPTR
    assert fwd_ex(L, None, None, None, N=0) == OK
    g = L.maxpool3d_bwd_ex
    # output sizes must be the window's: 6 with k3 s2 p1 gives 3
    assert g(x, i, y, 1, 1, 6, 6, 6, 4, 3, 3, 3, 3, 3, 2, 2, 2, 1, 1, 1, 1, 1, 1, 0, 0, 0, None, 0,
             None) == WINDOW
    assert g(x, i, y, 1, 1, 6, 6, 6, 3, 3, 3, 3, 3, 3, 2, 2, 2, 1, 1, 1, 1, 1, 1, 0, 0, 3, None, 0,
             None) == ALGO


def test_padded_plans(L):
    f32, f16 = torch.float32, torch.float16
    # padded or dilated: the depth walk for 16-bit types (clipped windows,
    # plane volume a multiple of 8), else the thread-per-output kernel
    assert mp.maxpool3d_fwd_ex_plan((2, 3, 8, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1),
                                    False, f16) == "fwd_roll"
    assert mp.maxpool3d_fwd_ex_plan((2, 3, 8, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1),
                                    False, f32) == "fwd_padded"
    assert mp.maxpool3d_fwd_ex_plan((2, 3, 7, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1),
                                    False, f16) == "fwd_padded"
    assert mp.maxpool3d_fwd_ex_plan((2, 3, 8, 9, 10), (2, 2, 2), (1, 1, 1), (0, 0, 0), (2, 1, 1),
                                    False, f32) == "fwd_padded"
    # backward: padding alone keeps the rolling ordered scatter, dilation
    # takes the direct gather
    out = mp.pool_out_size_ex((8, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1))
    assert mp.maxpool3d_bwd_ex_plan((2, 3, 8, 9, 10), out, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1),
                                    False, f16) == "bwd_overlap_roll"
    out_dl = mp.pool_out_size_ex((8, 9, 10), (2, 2, 2), (1, 1, 1), (0, 0, 0), (2, 1, 1))
    assert mp.maxpool3d_bwd_ex_plan((2, 3, 8, 9, 10), out_dl, (2, 2, 2), (1, 1, 1), (0, 0, 0), (2, 1, 1),
                                    False, f32) == "bwd_padded"
    assert mp.maxpool3d_bwd_ex_plan((2, 3, 8, 9, 10), out, (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1),
                                    False, f16, mp.BWD_ATOMIC) == "bwd_atomic"
    # the plain geometry keeps its fast paths
    assert mp.maxpool3d_fwd_ex_plan((2, 3, 16, 112, 112), (3, 3, 3), (2, 2, 2), (0, 0, 0), (1, 1, 1),
                                    False, f16) == "fwd_s2"
    assert mp.maxpool3d_bwd_ex_plan((2, 3, 16, 112, 112), (7, 55, 55), (3, 3, 3), (2, 2, 2), (0, 0, 0),
                                    (1, 1, 1), False, f16) == "bwd_overlap_roll"
    # ceil mode that adds a window is not the plain geometry
    assert mp.pool_out_size_ex((9, 9, 9), (2, 2, 2), (2, 2, 2), ceil_mode=True) == (5, 5, 5)
    assert mp.maxpool3d_fwd_ex_plan((1, 1, 9, 9, 9), (2, 2, 2), (2, 2, 2), (0, 0, 0), (1, 1, 1),
                                    True, f32) == "fwd_padded"


def _has_empty_window(I, K, S, p, dl, O):
    """Some window o < O has no position o*S - p + k*dl inside [0, I)."""
    return any(all(not (0 <= o * S - p + k * dl < I) for k in range(K)) for o in range(O))


def test_padded_out_size_matches_oracle(orc):
    # the library's size query (one axis at a time, the others of size 1)
    # against the oracle's; where the library refuses a geometry the oracle
    # sizes, a window must hold no input position
    for I in range(1, 12):
        for K in range(1, 5):
            for S in range(1, 4):
                for p in range(0, 3):
                    for dl in range(1, 4):
                        for cm in (False, True):
                            want = orc.ex_out_size(I, K, S, p, dl, cm)
                            try:
                                got = mp.pool_out_size_ex((I, 1, 1), (K, 1, 1), (S, 1, 1), (p, 0, 0),
                                                          (dl, 1, 1), cm)[0]
                            except mp.MP3DError as e:
                                assert e.status == WINDOW
                                assert want == 0 or _has_empty_window(I, K, S, p, dl, want), (
                                    I, K, S, p, dl, cm)
                                continue
                            assert got == want, (I, K, S, p, dl, cm)


def test_out_size_queries(L):
    od, oh, ow = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    r = (ctypes.byref(od), ctypes.byref(oh), ctypes.byref(ow))
    assert L.maxpool3d_out_size(16, 112, 112, 3, 3, 3, 2, 2, 2, *r) == OK
    assert (od.value, oh.value, ow.value) == (7, 55, 55)
    assert L.maxpool3d_out_size(32, 64, 64, 2, 2, 2, 2, 2, 2, *r) == OK
    assert (od.value, oh.value, ow.value) == (16, 32, 32)
    od.value = -5
    assert L.maxpool3d_out_size(4, 4, 4, 5, 2, 2, 1, 1, 1, *r) == WINDOW     # kernel > input
    assert L.maxpool3d_out_size(4, 4, 4, 2, 2, 2, 0, 1, 1, *r) == WINDOW     # stride 0
    assert L.maxpool3d_out_size(0, 4, 4, 2, 2, 2, 1, 1, 1, *r) == SHAPE
    assert L.maxpool3d_out_size(1 << 20, 1 << 11, 2, 1, 1, 1, 1, 1, 1, *r) == SHAPE   # volume 2^32
    assert od.value == -5                                                   # nothing stored
    assert L.maxpool3d_out_size(4, 4, 4, 2, 2, 2, 2, 2, 2, None, r[1], r[2]) == NULLPTR
    assert L.maxpool3d_ex_out_size(16, 56, 56, 3, 3, 3, 2, 2, 2, 1, 1, 1, 1, 1, 1, 0, *r) == OK
    assert (od.value, oh.value, ow.value) == (8, 28, 28)
    assert L.maxpool3d_ex_out_size(9, 9, 9, 2, 2, 2, 2, 2, 2, 0, 0, 0, 1, 1, 1, 1, *r) == OK
    assert (od.value, oh.value, ow.value) == (5, 5, 5)                      # ceil mode
    assert L.maxpool3d_ex_out_size(9, 9, 9, 2, 2, 2, 2, 2, 2, 2, 0, 0, 1, 1, 1, 0, *r) == WINDOW
    # the binding's helpers are the library's answers
    assert mp.pool_out_size((16, 112, 112), (3, 3, 3), (2, 2, 2)) == (7, 55, 55)
    with pytest.raises(mp.MP3DError):
        mp.pool_out_size((4, 4, 4), (5, 2, 2), (1, 1, 1))


def test_binding_has_no_size_arithmetic():
    # output sizes come from the library; the binding restates no formula
    src = open(os.path.join(ROOT, "bwd_maxpool3d_fwd_gb300", "__init__.py")).read()
    assert "//" not in src


def test_binding_checks_buffers_before_any_call():
    # wrong shapes and types raise before a pointer is handed over; these
    # tensors live on the CPU (no GPU here), so reaching the device check
    # would raise a different error
    x = torch.empty((2, 3, 8, 8, 8), dtype=torch.float16)
    y = torch.empty((2, 3, 4, 4, 4), dtype=torch.float16)
    idx = torch.empty((2, 3, 4, 4, 4), dtype=torch.int64)
    k = s = (2, 2, 2)
    with pytest.raises(ValueError, match="y: shape"):
        mp.maxpool3d_fwd(x, y[:, :, :3], idx, k, s)                      # short y
    with pytest.raises(TypeError, match="idx: dtype"):
        mp.maxpool3d_fwd(x, y, idx.int(), k, s)                          # int32 idx
    with pytest.raises(TypeError, match="y: dtype"):
        mp.maxpool3d_fwd(x, y.float(), idx, k, s)                        # y of another type
    with pytest.raises(ValueError, match="y: shape"):
        mp.adaptive_maxpool3d_fwd(x, y, idx, (4, 4, 3))
    with pytest.raises(ValueError, match="y: shape"):
        mp.maxpool3d_fwd_ex(x, y, idx, (3, 3, 3), (2, 2, 2))             # 3x3x3 outputs
    with pytest.raises(ValueError, match="CUDA"):
        mp.maxpool3d_fwd(x, y, idx, k, s)                                # all checks passed
    gin = torch.empty_like(x)
    with pytest.raises(TypeError, match="idx: dtype"):
        mp.maxpool3d_bwd(y, idx.int(), gin, k, s)
    with pytest.raises(ValueError, match="idx: shape"):
        mp.maxpool3d_bwd(y, idx[:1], gin, k, s)
    with pytest.raises(TypeError, match="grad_out: dtype"):
        mp.maxpool3d_bwd(y.float(), idx, gin, k, s)
    with pytest.raises(ValueError, match="the window gives"):
        mp.maxpool3d_bwd(y, idx, gin, (3, 3, 3), (2, 2, 2))
    with pytest.raises(ValueError, match="grad_out: shape"):
        mp.maxpool3d_bwd(y[:1], idx[:1], gin, k, s)                      # batch mismatch
    with pytest.raises(ValueError, match="x: shape"):
        mp.maxpool3d_bwd_recompute(x[:1], y, gin, k, s)
    with pytest.raises(ValueError, match="idx: shape"):
        mp.maxpool3d_bwd_noalloc(y, idx[:, :1], gin, k, s)
    xl = torch.empty((2, 8, 8, 8, 3), dtype=torch.float16)
    yl = torch.empty((2, 4, 4, 4, 3), dtype=torch.float16)
    with pytest.raises(ValueError, match="y: shape"):
        mp.maxpool3d_fwd_ndhwc(xl, yl[..., :2], None, k, s)
    with pytest.raises(ValueError, match="grad_out: shape"):
        mp.maxpool3d_bwd_ndhwc(yl[..., :2], idx, xl, k, s)
    with pytest.raises(ValueError, match="5-D"):
        mp.maxpool3d_fwd(x[0], y, idx, k, s)


def test_recompute_argument_errors_and_plans(L, bufs):
    x, g, gi, _ = bufs
    f = L.maxpool3d_bwd_recompute
    args = (1, 1, 4, 4, 4, 2, 2, 2, 2, 2, 2, 2, 2, 2, 0, None)
    assert f(None, g, gi, *args) == NULLPTR
    assert f(x, g, x + 8, *args) == ALIAS                 # grad_in overlaps x
    assert f(x, g, gi, 1, 1, 4, 4, 4, 3, 2, 2, 2, 2, 2, 2, 2, 2, 0, None) == WINDOW
    assert f(x, g, gi, 1, 1, 4, 4, 4, 2, 2, 2, 2, 2, 2, 2, 2, 2, 7, None) == DTYPE
    assert f(None, None, None, 0, 1, 4, 4, 4, 2, 2, 2, 2, 2, 2, 2, 2, 2, 0, None) == OK
    bf = torch.bfloat16
    assert mp.maxpool3d_bwd_recompute_plan((2, 3, 8, 8, 32), (4, 4, 16), (2, 2, 2), (2, 2, 2),
                                           bf) == "bwd_recompute_k2s2"
    assert mp.maxpool3d_bwd_recompute_plan((2, 3, 9, 8, 32), (4, 4, 16), (2, 2, 2), (2, 2, 2),
                                           bf) == "bwd_recompute_direct"
    assert mp.maxpool3d_bwd_recompute_plan((2, 3, 9, 9, 9), (4, 4, 4), (3, 3, 3), (2, 2, 2),
                                           bf) == "bwd_recompute_direct"
    assert mp.maxpool3d_bwd_recompute_plan((2, 3, 9, 9, 9), (4, 4, 4), None, None,
                                           bf) == "bwd_recompute_direct"


def test_path_names_cover_the_header():
    # every mp3d_path value the header declares has a name in the binding
    src = open(os.path.join(ROOT, "include", "mp3d.h")).read()
    values = {int(v) for v in re.findall(r"MP3D_PATH_\w+\s*=\s*(\d+)", src)}
    assert values and values == set(mp.PATHS), sorted(values ^ set(mp.PATHS))


def test_depth_walk_plans(L):
    f16, bf16, f32 = torch.float16, torch.bfloat16, torch.float32
    # the adaptive workload shape, both 16-bit types; fp32 keeps the slab
    for dt in (f16, bf16):
        assert mp.adaptive_maxpool3d_fwd_plan((2, 3, 30, 50, 50), (8, 12, 12), dt) == "fwd_roll"
    assert mp.adaptive_maxpool3d_fwd_plan((2, 3, 30, 50, 50), (8, 12, 12), f32) == "fwd_slab"
    # three windows over a depth slice (kernel 3, stride 1 along d): not the walk
    assert mp.maxpool3d_fwd_plan((1, 2, 8, 9, 10), (3, 2, 2), (1, 2, 2), f16) != "fwd_roll"
    # more outputs per depth than a CTA has threads: bands of output rows
    assert mp.adaptive_maxpool3d_fwd_plan((1, 2, 9, 40, 40), (4, 20, 20), f16) == "fwd_roll"
    # more than 65536 elements per slice: not the walk
    assert mp.adaptive_maxpool3d_fwd_plan((1, 1, 4, 300, 300), (2, 10, 10), f16) != "fwd_roll"


def test_wait_limit_setter_restores_the_default(L):
    f = L.mp3d_set_pipeline_wait_limit
    f.argtypes = [ctypes.c_int]
    f.restype = ctypes.c_int
    prev = f(5)
    try:
        assert f(-1) == 5
        assert f(-1) == 1 << 22
    finally:
        f(prev)


def test_no_undefined_symbols_of_the_library():
    # every function of the library's own namespace is defined in it
    import subprocess
    out = subprocess.run(["nm", "-DC", "--undefined-only", mp.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    assert "mp3d" not in out, out
