"""maxpool3d_bwd_noalloc: the backward for callers that cannot allocate
device memory while they run (engine plugins that own no allocator, fixed
memory budgets). It keeps its binary32 accumulators in a fixed array inside
the library instead of a caller workspace. Called here through the C ABI
(ctypes) and checked, within the atomic path's tolerance (1 ulp for
f16/bf16; 1e-6 of the sum of absolute contributions for f32), against the
oracle and against the existing entry point maxpool3d_bwd (its ordered
form, which the other tests hold bit-identical to the oracle), on several
calls in a row so that state left in the shared array by one call would
show in the next, up to exactly the array's limit.

This file is collected last on purpose."""
import ctypes

import pytest
import torch

import bwd_maxpool3d_fwd_gb300 as mp
import oracle
from gpu_helpers import DEV, ordered

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 8 << 20


def c_noalloc(g, idx, gin, kernel, stride):
    """Direct C-ABI call; returns the status code."""
    f = mp.lib().maxpool3d_bwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 5 + [ctypes.c_int] * 10 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    N, C, D, H, W = gin.shape
    od, oh, ow = g.shape[2:]
    k = kernel or (0, 0, 0)
    s = stride or (0, 0, 0)
    st = f(g.data_ptr(), idx.data_ptr(), gin.data_ptr(), N, C, D, H, W, od, oh, ow, *k, *s,
           mp.DTYPE_CODE[g.dtype], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st


def make_case(seed, dtype, in_shape, kernel=None, stride=None, out=None):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randint(-3, 4, in_shape, generator=gen).to(dtype).to(DEV)   # many ties
    if kernel is not None:
        out = mp.pool_out_size(in_shape[2:], kernel, stride)
    oshape = tuple(in_shape[:2]) + tuple(out)
    y = torch.empty(oshape, dtype=dtype, device=DEV)
    idx = torch.empty(oshape, dtype=torch.int64, device=DEV)
    if kernel is not None:
        mp.maxpool3d_fwd(x, y, idx, kernel, stride)
    else:
        mp.adaptive_maxpool3d_fwd(x, y, idx, out)
    g = torch.randn(oshape, generator=gen).to(dtype).to(DEV)
    return g, idx


def existing_entry_point(g, idx, in_shape, kernel, stride):
    gin = torch.empty(in_shape, dtype=g.dtype, device=DEV)
    mp.maxpool3d_bwd(g, idx, gin, kernel, stride)
    torch.cuda.synchronize()
    return gin


def oracle_grad_in(g, idx, in_shape):
    return oracle.maxpool3d_bwd(g.cpu(), idx.cpu(), tuple(in_shape[2:])).to(DEV)


def within_tolerance(a, b, g, idx):
    if a.dtype != torch.float32:
        return int((ordered(a) - ordered(b)).abs().max()) <= 1
    P = g.shape[0] * g.shape[1]
    vol = a[0, 0].numel()
    sabs = torch.zeros(a.numel(), dtype=torch.float64, device=DEV)
    flat = idx.reshape(P, -1) + (torch.arange(P, device=DEV) * vol).unsqueeze(1)
    sabs.index_add_(0, flat.reshape(-1), g.double().abs().reshape(-1))
    err = (a.double() - b.double()).abs().reshape(-1)
    return bool((err <= 1e-6 * sabs + 1e-30).all())


CASES = [
    (11, torch.float16, (2, 3, 9, 29, 117), (3, 3, 3), (2, 2, 2), None),
    (12, torch.bfloat16, (2, 2, 30, 50, 50), None, None, (8, 12, 12)),
    (13, torch.float32, (2, 3, 9, 29, 40), (3, 3, 3), (1, 2, 2), None),
    (14, torch.float16, (4, 8, 16, 112, 112), (3, 3, 3), (2, 2, 2), None),   # 6.4 Mi elements
    (15, torch.bfloat16, (1, 2, 16, 512, 512), (3, 3, 3), (2, 2, 2), None),  # exactly 8 Mi
]


def test_noalloc_matches_oracle_on_calls_in_a_row():
    # Several calls in a row with different shapes and types, then the
    # first case again: each must agree with the oracle and with the
    # workspace entry point, twice over.
    for seed, dtype, shape, k, s, out in CASES + CASES[:1]:
        g, idx = make_case(seed, dtype, shape, k, s, out)
        ref = oracle_grad_in(g, idx, shape)
        existing = existing_entry_point(g, idx, shape, k, s)
        for _ in range(2):
            gin = torch.full(shape, 3.0, dtype=dtype, device=DEV)
            assert c_noalloc(g, idx, gin, k, s) == 0
            assert within_tolerance(gin, ref, g, idx), ("oracle", seed, dtype, shape)
            assert within_tolerance(gin, existing, g, idx), ("maxpool3d_bwd", seed, dtype, shape)


def test_noalloc_rejects_problems_beyond_its_scratch():
    for shape, gshape, k in (((1, 1, 8, 1024, 1025), (1, 1, 4, 512, 512), (2, 2, 2)),
                             ((1, 1, 1, 3, 2796203), (1, 1, 1, 3, 1398101), (1, 1, 2))):
        n = shape[0] * shape[1] * shape[2] * shape[3] * shape[4]
        assert n > SCRATCH_LIMIT                       # 8 Mi + 1 in the second case
        gin = torch.full(shape, 3.0, dtype=torch.float16, device=DEV)
        g = torch.zeros(gshape, dtype=torch.float16, device=DEV)
        idx = torch.zeros(g.shape, dtype=torch.int64, device=DEV)
        assert c_noalloc(g, idx, gin, k, k) == 10     # MP3D_ERR_SCRATCH
        assert bool((gin == 3.0).all())                 # nothing written
    assert 1 * 1 * 1 * 3 * 2796203 == SCRATCH_LIMIT + 1
    # f32 accumulates in grad_in itself and is not limited by the scratch
    shape = (1, 1, 8, 1024, 1025)
    g32 = torch.zeros((1, 1, 4, 512, 512), dtype=torch.float32, device=DEV)
    idx = torch.zeros(g32.shape, dtype=torch.int64, device=DEV)
    gin32 = torch.empty(shape, dtype=torch.float32, device=DEV)
    assert c_noalloc(g32, idx, gin32, (2, 2, 2), (2, 2, 2)) == 0
    assert float(gin32.abs().max()) == 0.0
