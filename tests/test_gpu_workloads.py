"""The five workloads at full size, through the same entry points the
benchmark times (needs a GPU). Workloads 0, 1, 2 and 4 are compared with
the oracle in full; workload 3 (822M inputs) on a sample of planes, plus
properties checked on every output. The padded workload the benchmark also
times is compared in full."""
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


def test_workload3_sampled_and_properties():
    w = workloads.WORKLOADS[3]
    x, g = workloads.make_x(w), workloads.make_grad_out(w)
    xd = x.to(DEV)
    y, idx, gin = run(w, xd, g.to(DEV))
    P, vol = w.planes, w.D * w.H * w.W
    # every output: y is a bit copy of the input at idx, idx lies in its window
    yb = bits(y).reshape(P, -1)
    xb = bits(xd).reshape(P, vol)
    assert torch.equal(yb, torch.gather(xb, 1, idx.reshape(P, -1)))
    HW = w.H * w.W
    d, h, ww = idx // HW, (idx % HW) // w.W, idx % w.W
    od = torch.arange(w.out[0], device=DEV).view(1, 1, -1, 1, 1)
    oh = torch.arange(w.out[1], device=DEV).view(1, 1, 1, -1, 1)
    ow = torch.arange(w.out[2], device=DEV).view(1, 1, 1, 1, -1)
    for c, o, k, s in ((d, od, 3, 2), (h, oh, 3, 2), (ww, ow, 3, 2)):
        assert bool(((c >= o * s) & (c < o * s + k)).all())
    # ties at the maximum are present in this workload (first occurrence matters)
    # sampled planes against the oracle, forward and backward
    planes = [0, 1, 63, 64, 1000, 2047, 2048, 3071, 4094, 4095]
    xs = x.reshape(P, w.D, w.H, w.W)[planes].reshape(1, len(planes), w.D, w.H, w.W).contiguous()
    gs = g.reshape(P, *w.out)[planes].reshape(1, len(planes), *w.out).contiguous()
    y_ref, i_ref = oracle.maxpool3d_fwd(xs, w.kernel, w.stride)
    gin_ref = oracle.maxpool3d_bwd(gs, i_ref, (w.D, w.H, w.W))
    sel = torch.tensor(planes, device=DEV)
    assert torch.equal(idx.reshape(P, -1)[sel].cpu(), i_ref.reshape(len(planes), -1))
    assert_bits_equal(y.reshape(P, -1)[sel].cpu(), y_ref.reshape(len(planes), -1), "y")
    assert_bits_equal(gin.reshape(P, -1)[sel].cpu(), gin_ref.reshape(len(planes), -1), "grad_in")
    # the tie injection produced windows whose maximum occurs more than once
    win = xs.float().unfold(2, 3, 2).unfold(3, 3, 2).unfold(4, 3, 2).reshape(
        len(planes), *w.out, 27)
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
