"""Seeded synthetic inputs for the five pooling workloads.

This module holds the workload table (shapes, types and windows as stated
for each workload) and the seeded generators that fill the input and the
upstream gradient. It contains none of the pooling arithmetic: output sizes
are the stated constants of each workload (the CUDA library and the oracle
each compute their own, and the tests check both against these), and no
generator looks at window maxima.

Data is produced on the CPU with ``torch.Generator`` in fixed chunks of
planes, each chunk with its own seed, so that any plane can be regenerated
alone (used for sampled checks) and chunks can be filled in parallel.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import torch

PLANES_PER_CHUNK = 64
BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str                  # "adaptive" or "fixed"
    dtype: torch.dtype
    N: int
    C: int
    D: int
    H: int
    W: int
    out: tuple                 # stated output size (OD, OH, OW)
    kernel: tuple = (0, 0, 0)  # fixed windows only
    stride: tuple = (0, 0, 0)
    x_recipe: str = "normal"   # "perm", "uniform", "normal", "normal_dup5"
    g_recipe: str = "normal"
    seed: int = BASE_SEED
    pad: tuple = (0, 0, 0)     # fixed windows: padding per side (output sizes as stated)

    @property
    def planes(self) -> int:
        return self.N * self.C

    @property
    def in_shape(self):
        return (self.N, self.C, self.D, self.H, self.W)

    @property
    def out_shape(self):
        return (self.N, self.C) + tuple(self.out)

    @property
    def elem_bytes(self) -> int:
        return torch.empty((), dtype=self.dtype).element_size()


WORKLOADS = [
    # 0: adaptive fp32, 2x3x8^3 -> 4^3 (divisible: disjoint windows).
    Workload("adaptive_f32_2x3x8x8x8_to_4x4x4", "adaptive", torch.float32,
             2, 3, 8, 8, 8, (4, 4, 4), x_recipe="perm", seed=BASE_SEED + 0),
    # 1: adaptive fp16, 16x64x30x50x50 -> 8x12x12 (overlapping windows).
    Workload("adaptive_f16_16x64x30x50x50_to_8x12x12", "adaptive", torch.float16,
             16, 64, 30, 50, 50, (8, 12, 12), x_recipe="uniform", seed=BASE_SEED + 1),
    # 2: fixed bf16, kernel 2^3 stride 2, 8x64x32x64x64 -> 16x32x32 (disjoint).
    Workload("fixed_k2s2_bf16_8x64x32x64x64", "fixed", torch.bfloat16,
             8, 64, 32, 64, 64, (16, 32, 32), (2, 2, 2), (2, 2, 2),
             x_recipe="normal", seed=BASE_SEED + 2),
    # 3: fixed fp16, kernel 3^3 stride 2, 32x128x16x112x112 -> 7x55x55
    #    (overlapping), 5% of values duplicated within windows.
    Workload("fixed_k3s2_f16_32x128x16x112x112", "fixed", torch.float16,
             32, 128, 16, 112, 112, (7, 55, 55), (3, 3, 3), (2, 2, 2),
             x_recipe="normal_dup5", seed=BASE_SEED + 3),
    # 4: adaptive fp32 global pool, 64x512x8x14x14 -> 1x1x1.
    Workload("adaptive_global_f32_64x512x8x14x14", "adaptive", torch.float32,
             64, 512, 8, 14, 14, (1, 1, 1), x_recipe="uniform", seed=BASE_SEED + 4),
]


# Further workloads the benchmark can time (not among the five above): the
# k3s2 workload's input with padding 1 on every side, 3x3x3 windows, stride
# 2 -> 8x56x56 outputs.
EXTRA = [
    Workload("fixed_k3s2p1_f16_32x128x16x112x112", "fixed", torch.float16,
             32, 128, 16, 112, 112, (8, 56, 56), (3, 3, 3), (2, 2, 2),
             x_recipe="normal_dup5", seed=BASE_SEED + 3, pad=(1, 1, 1)),
]


def by_name_or_index(key) -> Workload:
    """A workload of WORKLOADS by index, or of WORKLOADS + EXTRA by name."""
    if isinstance(key, int) or str(key).isdigit():
        return WORKLOADS[int(key)]
    for w in WORKLOADS + EXTRA:
        if w.name == key:
            return w
    raise KeyError(f"no workload {key!r}")


def _chunk_seed(seed: int, chunk: int, stream: int) -> int:
    return (seed * 1_000_003 + stream * 7_919 * 65_537 + chunk) & 0x7FFF_FFFF_FFFF


def _fill_x(w: Workload, chunk: int, nplanes: int) -> torch.Tensor:
    gen = torch.Generator().manual_seed(_chunk_seed(w.seed, chunk, 0))
    shape = (nplanes, w.D, w.H, w.W)
    if w.x_recipe == "perm":
        # A random permutation of distinct values, scaled to [-1, 1).
        n = nplanes * w.D * w.H * w.W
        perm = torch.randperm(n, generator=gen, dtype=torch.float64)
        return (perm * (2.0 / n) - 1.0).to(w.dtype).reshape(shape)
    if w.x_recipe == "uniform":
        return (torch.rand(shape, generator=gen) * 2.0 - 1.0).to(w.dtype)
    if w.x_recipe in ("normal", "normal_dup5"):
        x = torch.randn(shape, generator=gen).to(w.dtype)
        if w.x_recipe == "normal_dup5":
            # Duplicate a seeded 5% of the values into their W-neighbour.
            # For stride-2 size-3 windows every pair (w, w+1) lies inside a
            # common window, so each copy repeats a value inside a window;
            # where the copied value is that window's maximum it makes a tie
            # at the maximum.
            pick = torch.rand((nplanes, w.D, w.H, w.W - 1), generator=gen) < 0.05
            src = x[..., :-1].clone()
            x[..., 1:] = torch.where(pick, src, x[..., 1:])
        return x
    raise ValueError(w.x_recipe)


def _fill_g(w: Workload, chunk: int, nplanes: int) -> torch.Tensor:
    gen = torch.Generator().manual_seed(_chunk_seed(w.seed, chunk, 1))
    shape = (nplanes,) + tuple(w.out)
    return torch.randn(shape, generator=gen).to(w.dtype)


def _generate(w: Workload, fill, per_plane_shape, planes=None, threads=None):
    """Fill whole chunks in parallel, then keep the requested planes."""
    nchunks = (w.planes + PLANES_PER_CHUNK - 1) // PLANES_PER_CHUNK
    if planes is None:
        chunks = list(range(nchunks))
    else:
        chunks = sorted({int(p) // PLANES_PER_CHUNK for p in planes})

    def one(c):
        n = min(PLANES_PER_CHUNK, w.planes - c * PLANES_PER_CHUNK)
        return c, fill(w, c, n)

    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(max_workers=threads) as ex:
        parts = dict(ex.map(one, chunks))
    if planes is None:
        out = torch.cat([parts[c] for c in chunks], dim=0)
        return out.reshape((w.N, w.C) + per_plane_shape)
    rows = [parts[int(p) // PLANES_PER_CHUNK][int(p) % PLANES_PER_CHUNK] for p in planes]
    return torch.stack(rows, dim=0).reshape((1, len(rows)) + per_plane_shape)


def make_x(w: Workload, planes=None) -> torch.Tensor:
    """Input x as a contiguous CPU tensor (N, C, D, H, W). With `planes` (flat
    plane indices n*C + c) only those planes, shaped (1, len(planes), D, H, W)."""
    return _generate(w, _fill_x, (w.D, w.H, w.W), planes).contiguous()


def make_grad_out(w: Workload, planes=None) -> torch.Tensor:
    """Upstream gradient, shaped like the stated output (N, C, OD, OH, OW)."""
    return _generate(w, _fill_g, tuple(w.out), planes).contiguous()
