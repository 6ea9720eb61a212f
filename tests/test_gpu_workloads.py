"""The five workloads at full size, through the same entry points the
benchmark times (needs a GPU), compared with the oracle in full: indices,
output bits and grad_in bits of every plane. Workload 3 (822M inputs) is
checked in chunks of planes on a thread pool. The padded workload the
benchmark also times is compared in full, and workload 3 in the
channels-last layout on sampled planes."""
import concurrent.futures as cf
import os

import pytest
import torch

import bwd_maxpool3d_fwd_gb300 as mp
import oracle
from bwd_maxpool3d_fwd_gb300 import workloads
from gpu_helpers import DEV, assert_bits_equal, bits, ordered

pytestmark = pytest.mark.gpu


def run(w, x_dev, g_dev, algo=mp.BWD_AUTO):
    y = torch.empty(w.out_shape, dtype=w.dtype, device=DEV)
    idx = torch.empty(w.out_shape, dtype=torch.int64, device=DEV)
    if w.mode == "fixed":
        mp.maxpool3d_fwd(x_dev, y, idx, w.kernel, w.stride)
        k, s = w.kernel, w.stride
    else:
        mp.adaptive_maxpool3d_fwd(x_dev, y, idx, w.out)
        k = s = None
    gin = torch.empty(w.in_shape, dtype=w.dtype, device=DEV)
    nbytes = mp.maxpool3d_bwd_workspace_bytes(w.in_shape, w.dtype, algo)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=DEV) if nbytes else None
    mp.maxpool3d_bwd(g_dev, idx, gin, k, s, algo=algo, workspace=ws)
    torch.cuda.synchronize()
    return y, idx, gin


def oracle_fwd(w, x):
    if w.mode == "fixed":
        return oracle.maxpool3d_fwd(x, w.kernel, w.stride)
    return oracle.adaptive_maxpool3d_fwd(x, w.out)


@pytest.mark.parametrize("n", [0, 1, 2, 4])
def test_workload_full(n):
    w = workloads.WORKLOADS[n]
    x, g = workloads.make_x(w), workloads.make_grad_out(w)
    y_ref, i_ref = oracle_fwd(w, x)
    assert tuple(y_ref.shape[2:]) == tuple(w.out)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, (w.D, w.H, w.W))
    y, idx, gin = run(w, x.to(DEV), g.to(DEV))
    assert torch.equal(idx.cpu(), i_ref)
    assert_bits_equal(y.cpu(), y_ref, "y")
    assert_bits_equal(gin.cpu(), gin_ref, "grad_in")


def test_workload1_atomic_ablation():
    w = workloads.WORKLOADS[1]
    x, g = workloads.make_x(w), workloads.make_grad_out(w)
    _, i_ref = oracle_fwd(w, x)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, (w.D, w.H, w.W))
    _, _, gin = run(w, x.to(DEV), g.to(DEV), algo=mp.BWD_ATOMIC)
    assert int((ordered(gin.cpu()) - ordered(gin_ref)).abs().max()) <= 1


def _oracle_chunk_matches(w, x, g, y, idx, gin, p0, p1):
    """Planes [p0, p1) of the GPU results against the oracle, bit for bit."""
    n = p1 - p0
    xs = x.reshape(w.planes, w.D, w.H, w.W)[p0:p1].reshape(1, n, w.D, w.H, w.W)
    gs = g.reshape(w.planes, *w.out)[p0:p1].reshape(1, n, *w.out)
    y_ref, i_ref = oracle.maxpool3d_fwd(xs, w.kernel, w.stride)
    gin_ref = oracle.maxpool3d_bwd(gs, i_ref, (w.D, w.H, w.W))
    ok_i = torch.equal(idx.reshape(w.planes, -1)[p0:p1], i_ref.reshape(n, -1))
    ok_y = torch.equal(bits(y.reshape(w.planes, -1)[p0:p1]), bits(y_ref.reshape(n, -1)))
    ok_g = torch.equal(bits(gin.reshape(w.planes, -1)[p0:p1]), bits(gin_ref.reshape(n, -1)))
    return p0, ok_i, ok_y, ok_g


def test_workload3_full():
    # the k3s2 fp16 workload (4096 planes, 822M inputs) in full: idx, y bits
    # and grad_in bits of every plane against the oracle, in chunks of planes
    # checked by a thread pool (the oracle releases the GIL in its C calls)
    w = workloads.WORKLOADS[3]
    x, g = workloads.make_x(w), workloads.make_grad_out(w)
    y, idx, gin = run(w, x.to(DEV), g.to(DEV))
    y, idx, gin = y.cpu(), idx.cpu(), gin.cpu()
    chunk = 64
    bounds = [(p, min(p + chunk, w.planes)) for p in range(0, w.planes, chunk)]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda b: _oracle_chunk_matches(w, x, g, y, idx, gin, *b), bounds))
    bad = [r for r in results if not all(r[1:])]
    assert not bad, f"planes differing from the oracle (first plane of chunk, idx, y, grad_in): {bad[:4]}"
    # values only (idx NULL, compiled without the winners' codes): the same y
    # bits as the forward with indices, on every plane
    yv = torch.empty(w.out_shape, dtype=w.dtype, device=DEV)
    mp.maxpool3d_fwd(x.to(DEV), yv, None, w.kernel, w.stride)
    torch.cuda.synchronize()
    assert torch.equal(bits(yv.cpu()), bits(y))
    # the tie injection produced windows whose maximum occurs more than once
    planes = [0, 1, 2047, 4095]
    xs = x.reshape(w.planes, w.D, w.H, w.W)[planes].float()
    win = xs.unfold(1, 3, 2).unfold(2, 3, 2).unfold(3, 3, 2).reshape(len(planes), *w.out, 27)
    repeats = (win == win.max(dim=-1, keepdim=True).values).sum(-1)
    assert int((repeats > 1).sum()) > 0.01 * repeats.numel()


def test_padded_workload_full():
    # the padded workload the benchmark times (3x3x3, stride 2, padding 1,
    # fp16, 8x64x16x56x56), forward and backward in full against the oracle
    shape, k, s, p, dl = (8, 64, 16, 56, 56), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1)
    gen = torch.Generator().manual_seed(20261302)
    x = torch.randn(shape, generator=gen).half()
    y_ref, i_ref = oracle.maxpool3d_fwd_ex(x, k, s, p, dl, False)
    g = torch.randn(y_ref.shape, generator=gen).half()
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    xd, gd = x.to(DEV), g.to(DEV)
    y = torch.empty(y_ref.shape, dtype=x.dtype, device=DEV)
    idx = torch.empty(y_ref.shape, dtype=torch.int64, device=DEV)
    gin = torch.empty(shape, dtype=x.dtype, device=DEV)
    mp.maxpool3d_fwd_ex(xd, y, idx, k, s, p, dl)
    mp.maxpool3d_bwd_ex(gd, idx, gin, k, s, p, dl)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), i_ref)
    assert_bits_equal(y.cpu(), y_ref, "y (padded workload)")
    assert_bits_equal(gin.cpu(), gin_ref, "grad_in (padded workload)")


def test_padded_large_workload_full():
    # 3x3x3 windows, stride 2, padding 1 at the size of the k3s2 workload
    # (its input, ties included), forward and backward on every plane
    # against the oracle, checked in chunks of planes on a thread pool
    w = workloads.WORKLOADS[3]
    k, s, p = (3, 3, 3), (2, 2, 2), (1, 1, 1)
    x = workloads.make_x(w)
    out = mp.pool_out_size_ex((w.D, w.H, w.W), k, s, p)
    gen = torch.Generator().manual_seed(20261303)
    g = torch.randn((w.N, w.C) + out, generator=gen).half()
    xd, gd = x.to(DEV), g.to(DEV)
    y = torch.empty(g.shape, dtype=torch.float16, device=DEV)
    idx = torch.empty(g.shape, dtype=torch.int64, device=DEV)
    gin = torch.empty(w.in_shape, dtype=torch.float16, device=DEV)
    assert mp.maxpool3d_fwd_ex_plan(w.in_shape, k, s, p, (1, 1, 1), False, torch.float16) == "fwd_s2"
    mp.maxpool3d_fwd_ex(xd, y, idx, k, s, p)
    mp.maxpool3d_bwd_ex(gd, idx, gin, k, s, p)
    torch.cuda.synchronize()
    y, idx, gin = y.cpu(), idx.cpu(), gin.cpu()
    del xd, gd
    P = w.planes

    def chunk(b):
        p0, p1 = b
        n = p1 - p0
        xs = x.reshape(P, w.D, w.H, w.W)[p0:p1].reshape(1, n, w.D, w.H, w.W)
        gs = g.reshape(P, *out)[p0:p1].reshape(1, n, *out)
        y_ref, i_ref = oracle.maxpool3d_fwd_ex(xs, k, s, p, (1, 1, 1), False)
        gin_ref = oracle.maxpool3d_bwd(gs, i_ref, (w.D, w.H, w.W))
        return (p0, torch.equal(idx.reshape(P, -1)[p0:p1], i_ref.reshape(n, -1)),
                torch.equal(bits(y.reshape(P, -1)[p0:p1]), bits(y_ref.reshape(n, -1))),
                torch.equal(bits(gin.reshape(P, -1)[p0:p1]), bits(gin_ref.reshape(n, -1))))

    bounds = [(q, min(q + 64, P)) for q in range(0, P, 64)]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = list(ex.map(chunk, bounds))
    bad = [r for r in results if not all(r[1:])]
    assert not bad, f"planes differing from the oracle (first plane of chunk, idx, y, grad_in): {bad[:4]}"


def test_workload3_channels_last_sampled():
    # the k3s2 fp16 workload in the channels-last layout (32 x 16 x 112 x 112
    # x 128, the same values with the channel axis last) through the
    # channels-last forward and backward the benchmark times; every (n, c)
    # plane of the first and last sample and 128 seeded others are compared
    # with the oracle in full (idx, y bits, grad_in bits)
    w = workloads.WORKLOADS[3]
    k, s = w.kernel, w.stride
    assert mp.maxpool3d_bwd_ndhwc_plan(w.in_shape, w.out, k, s, torch.float16) == "bwd_ndhwc_roll"
    x, g = workloads.make_x(w), workloads.make_grad_out(w)
    xl = x.permute(0, 2, 3, 4, 1).contiguous().to(DEV)
    gl = g.permute(0, 2, 3, 4, 1).contiguous().to(DEV)
    oshape = (w.N,) + tuple(w.out) + (w.C,)
    y = torch.empty(oshape, dtype=w.dtype, device=DEV)
    idx = torch.empty(oshape, dtype=torch.int64, device=DEV)
    gin = torch.empty_like(xl)
    mp.maxpool3d_fwd_ndhwc(xl, y, idx, k, s)
    mp.maxpool3d_bwd_ndhwc(gl, idx, gin, k, s)
    torch.cuda.synchronize()
    y, idx, gin = y.cpu(), idx.cpu(), gin.cpu()
    del xl, gl
    gen = torch.Generator().manual_seed(20261304)
    planes = [(0, c) for c in range(w.C)] + [(w.N - 1, c) for c in range(w.C)]
    planes += [(int(n), int(c)) for n, c in zip(torch.randint(1, w.N - 1, (128,), generator=gen),
                                                torch.randint(0, w.C, (128,), generator=gen))]

    def chunk(b):
        sel = planes[b[0]:b[1]]
        ns = torch.tensor([p[0] for p in sel])
        cs = torch.tensor([p[1] for p in sel])
        xs = x[ns, cs].unsqueeze(0)                       # (1, P, D, H, W)
        gs = g[ns, cs].unsqueeze(0)
        y_ref, i_ref = oracle.maxpool3d_fwd(xs, k, s)
        gin_ref = oracle.maxpool3d_bwd(gs, i_ref, (w.D, w.H, w.W))
        return (b[0], torch.equal(idx[ns, ..., cs], i_ref[0]),
                torch.equal(bits(y[ns, ..., cs]), bits(y_ref[0])),
                torch.equal(bits(gin[ns, ..., cs]), bits(gin_ref[0])))

    bounds = [(q, min(q + 32, len(planes))) for q in range(0, len(planes), 32)]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = list(ex.map(chunk, bounds))
    bad = [r for r in results if not all(r[1:])]
    assert not bad, f"sampled planes differing from the oracle (first of chunk, idx, y, grad_in): {bad[:4]}"
