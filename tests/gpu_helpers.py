"""Shared helpers for the GPU parity tests: run the CUDA path through the
C ABI binding and compare with the oracle bit for bit."""
from __future__ import annotations

import torch

import bwd_maxpool3d_fwd_gb300 as mp

DEV = torch.device("cuda:0")
DTYPES = (torch.float32, torch.float16, torch.bfloat16)


def bits(t: torch.Tensor) -> torch.Tensor:
    t = t.contiguous()
    return t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)


def gpu_fwd(x_cpu, kernel=None, stride=None, out_size=None):
    """Forward on the GPU; returns (y, idx) on the CPU."""
    x = x_cpu.to(DEV)
    if kernel is not None:
        out = mp.pool_out_size(x.shape[2:], kernel, stride)
    else:
        out = tuple(out_size)
    y = torch.empty(x.shape[:2] + out, dtype=x.dtype, device=DEV)
    idx = torch.empty(x.shape[:2] + out, dtype=torch.int64, device=DEV)
    if kernel is not None:
        mp.maxpool3d_fwd(x, y, idx, kernel, stride)
    else:
        mp.adaptive_maxpool3d_fwd(x, y, idx, out_size)
    torch.cuda.synchronize()
    return y.cpu(), idx.cpu()


def gpu_bwd(g_cpu, idx_cpu, in_shape, kernel=None, stride=None, algo=mp.BWD_AUTO, offset=0):
    """Backward on the GPU; returns grad_in on the CPU. offset > 0 places
    grad_in that many elements past a 16-byte boundary (paths that need
    aligned 16-byte stores then give way to the others)."""
    g = g_cpu.to(DEV)
    idx = idx_cpu.to(DEV)
    n = 1
    for v in in_shape:
        n *= v
    gin = torch.empty(n + offset, dtype=g.dtype, device=DEV)[offset:].view(in_shape)
    ws = None
    nbytes = mp.maxpool3d_bwd_workspace_bytes(in_shape, g.dtype, algo)
    if nbytes:
        ws = torch.empty(nbytes // 4, dtype=torch.float32, device=DEV)
    mp.maxpool3d_bwd(g, idx, gin, kernel, stride, algo=algo, workspace=ws)
    torch.cuda.synchronize()
    return gin.cpu()


def random_input(gen, shape, dtype, kind):
    """Test inputs: 'normal', 'ties' (small integers, many equal maxima),
    'special' (ties plus +-0, +-inf and NaNs)."""
    if kind == "normal":
        return torch.randn(shape, generator=gen).to(dtype)
    x = torch.randint(-3, 4, shape, generator=gen).float()
    if kind == "special":
        r = torch.rand(shape, generator=gen)
        x = torch.where(r < 0.10, torch.tensor(-0.0), x)
        x = torch.where((r >= 0.10) & (r < 0.15), torch.tensor(0.0), x)
        x = torch.where((r >= 0.15) & (r < 0.16), torch.tensor(float("inf")), x)
        x = torch.where((r >= 0.16) & (r < 0.17), torch.tensor(float("-inf")), x)
        x = torch.where((r >= 0.17) & (r < 0.18), torch.tensor(float("nan")), x)
    return x.to(dtype)


def ordered(t: torch.Tensor) -> torch.Tensor:
    """Bit patterns mapped to integers in value order (adjacent values of the
    type differ by 1; +0 and -0 both map to 0)."""
    b = bits(t).long()
    w = 32 if t.element_size() == 4 else 16
    b = b & ((1 << w) - 1)
    sign = b >> (w - 1)
    mag = b & ((1 << (w - 1)) - 1)
    return torch.where(sign == 1, -mag, mag)


def assert_bits_equal(a: torch.Tensor, b: torch.Tensor, what: str):
    ba, bb = bits(a).reshape(-1), bits(b).reshape(-1)
    if not torch.equal(ba, bb):
        bad = torch.nonzero(ba != bb).reshape(-1)
        # NaN payloads are not pinned: two NaNs count as equal.
        fa, fb = a.float().reshape(-1)[bad], b.float().reshape(-1)[bad]
        real = bad[~(torch.isnan(fa) & torch.isnan(fb))]
        assert real.numel() == 0, (
            f"{what}: {real.numel()} elements differ; first at {real[:5].tolist()}: "
            f"{a.reshape(-1)[real[:5]].tolist()} vs {b.reshape(-1)[real[:5]].tolist()}")

