"""CUDA path against the oracle, element by element (needs a GPU).

Forward values and indices, and the gather backward, must match the oracle
bit for bit; the atomic ablation must be within 1e-6 of the sum of the
absolute contributions (f32) or 1 ulp (f16, bf16)."""
import pytest
import torch

import bwd_maxpool3d_fwd_gb300 as mp
import oracle
from gpu_helpers import (DEV, DTYPES, assert_bits_equal, bits, gpu_bwd, gpu_fwd, ordered,
                         random_input)

pytestmark = pytest.mark.gpu

KINDS = ("normal", "ties", "special")


def _fixed_cases(seed, n):
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(n):
        k = [int(v) for v in torch.randint(1, 5, (3,), generator=g)]
        s = [int(v) for v in torch.randint(1, 4, (3,), generator=g)]
        D = k[0] + int(torch.randint(0, 14, (1,), generator=g))
        H = k[1] + int(torch.randint(0, 40, (1,), generator=g))
        W = k[2] + int(torch.randint(0, 150, (1,), generator=g))
        out.append((tuple(k), tuple(s), (2, 3, D, H, W)))
    return out


# Workload-like windows on shapes that span several tiles plus ragged tails.
FIXED_CASES = [
    ((2, 2, 2), (2, 2, 2), (2, 3, 9, 37, 70)),
    ((3, 3, 3), (2, 2, 2), (2, 3, 9, 29, 117)),
    ((3, 3, 3), (2, 2, 2), (1, 2, 16, 112, 112)),
    ((2, 2, 2), (2, 2, 2), (1, 2, 32, 64, 64)),
    ((3, 3, 3), (1, 1, 1), (1, 2, 6, 20, 33)),
    ((1, 1, 1), (1, 1, 1), (1, 2, 3, 5, 7)),
    ((2, 3, 1), (3, 2, 4), (2, 2, 11, 13, 17)),
] + _fixed_cases(101, 24)


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(FIXED_CASES)))
def test_fixed_fwd_bwd(case, dtype):
    k, s, shape = FIXED_CASES[case]
    gen = torch.Generator().manual_seed(1000 + case)
    kind = KINDS[case % 3]
    x = random_input(gen, shape, dtype, kind)
    y_ref, i_ref = oracle.maxpool3d_fwd(x, k, s)
    y, idx = gpu_fwd(x, kernel=k, stride=s)
    assert torch.equal(idx, i_ref), f"idx differs ({k}, {s}, {shape}, {kind})"
    assert_bits_equal(y, y_ref, "y")
    g = torch.randn(y_ref.shape, generator=gen).to(dtype)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    gin = gpu_bwd(g, i_ref, shape, k, s)
    assert_bits_equal(gin, gin_ref, "grad_in")


def _adaptive_cases():
    g = torch.Generator().manual_seed(202)
    out = [((2, 3, 8, 8, 8), (4, 4, 4)), ((2, 3, 30, 50, 50), (8, 12, 12)),
           ((1, 3, 8, 14, 14), (1, 1, 1)), ((1, 1, 7, 7, 7), (8, 8, 8)),
           ((2, 2, 7, 7, 7), (3, 3, 3)), ((1, 2, 10, 10, 10), (3, 4, 6)),
           ((1, 1, 3, 5, 9), (7, 9, 12))]
    for _ in range(14):
        I = [int(v) for v in torch.randint(1, 40, (3,), generator=g)]
        O = [int(torch.randint(1, i + 4, (1,), generator=g)) for i in I]
        out.append(((2, 2) + tuple(I), tuple(O)))
    return out


ADAPTIVE_CASES = _adaptive_cases()


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(ADAPTIVE_CASES)))
def test_adaptive_fwd_bwd(case, dtype):
    shape, out = ADAPTIVE_CASES[case]
    gen = torch.Generator().manual_seed(2000 + case)
    kind = KINDS[case % 3]
    x = random_input(gen, shape, dtype, kind)
    y_ref, i_ref = oracle.adaptive_maxpool3d_fwd(x, out)
    y, idx = gpu_fwd(x, out_size=out)
    assert torch.equal(idx, i_ref), f"idx differs ({shape} -> {out}, {kind})"
    assert_bits_equal(y, y_ref, "y")
    g = torch.randn(y_ref.shape, generator=gen).to(dtype)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    gin = gpu_bwd(g, i_ref, shape)
    assert_bits_equal(gin, gin_ref, "grad_in")


def _atomic_tolerance_ok(gin, gin_ref, g, idx, dtype):
    if dtype == torch.float32:
        P = g.shape[0] * g.shape[1]
        sabs = torch.zeros(gin.numel(), dtype=torch.float64)
        flat_idx = idx.reshape(P, -1) + (torch.arange(P) * gin[0, 0].numel()).unsqueeze(1)
        sabs.index_add_(0, flat_idx.reshape(-1), g.double().abs().reshape(-1))
        err = (gin.double().reshape(-1) - gin_ref.double().reshape(-1)).abs()
        return bool((err <= 1e-6 * sabs + 1e-30).all())
    return bool(((ordered(gin) - ordered(gin_ref)).abs() <= 1).all())


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", [1, 2, 4, 7, 9])
def test_atomic_ablation(case, dtype):
    k, s, shape = FIXED_CASES[case]
    gen = torch.Generator().manual_seed(3000 + case)
    x = random_input(gen, shape, dtype, "ties")
    _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    g = torch.randn(i_ref.shape, generator=gen).to(dtype)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    gin = gpu_bwd(g, i_ref, shape, k, s, algo=mp.BWD_ATOMIC)
    assert _atomic_tolerance_ok(gin, gin_ref, g, i_ref, dtype)


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
def test_gather_is_deterministic(dtype):
    k, s, shape = FIXED_CASES[1]
    gen = torch.Generator().manual_seed(77)
    x = random_input(gen, shape, dtype, "ties")
    _, idx = oracle.maxpool3d_fwd(x, k, s)
    g = torch.randn(idx.shape, generator=gen).to(dtype)
    first = bits(gpu_bwd(g, idx, shape, k, s))
    for _ in range(5):
        assert torch.equal(bits(gpu_bwd(g, idx, shape, k, s)), first)


def test_gpu_roundings_match_oracle_conversions():
    # binary32 -> binary16 / bfloat16 rounding of the CUDA path (exercised
    # through an overlap sum of two terms) against the oracle's encoders.
    gen = torch.Generator().manual_seed(9)
    for dtype, enc in ((torch.float16, oracle.f32_to_f16), (torch.bfloat16, oracle.f32_to_bf16)):
        n = 4096
        a = torch.randn(n, generator=gen).to(dtype)
        b = (torch.randn(n, generator=gen) * 1e-3).to(dtype)
        g = torch.stack([a, b], dim=1).reshape(n, 1, 1, 1, 2)
        idx = torch.ones_like(g, dtype=torch.int64)
        gin = gpu_bwd(g.contiguous(), idx, (n, 1, 1, 1, 3), (1, 1, 2), (1, 1, 1))
        got = bits(gin[:, 0, 0, 0, 1]).long() & 0xFFFF
        s32 = a.float() + b.float()                       # the binary32 sum
        want = torch.tensor([enc(float(v)) for v in s32])
        assert torch.equal(got, want.long())


def test_empty_input_is_noop():
    x = torch.empty((0, 3, 4, 4, 4), device=DEV)
    y = torch.empty((0, 3, 2, 2, 2), device=DEV)
    idx = torch.empty((0, 3, 2, 2, 2), dtype=torch.int64, device=DEV)
    mp.maxpool3d_fwd(x, y, idx, (2, 2, 2), (2, 2, 2))
    mp.maxpool3d_bwd(y, idx, x, (2, 2, 2), (2, 2, 2))
    torch.cuda.synchronize()


def test_unaligned_pointers_take_scalar_paths():
    # Views that start one element into a buffer: not 16-byte aligned.
    gen = torch.Generator().manual_seed(31)
    for dtype in DTYPES:
        shape, k, s = (2, 3, 9, 17, 40), (3, 3, 3), (2, 2, 2)
        x = random_input(gen, shape, dtype, "ties")
        y_ref, i_ref = oracle.maxpool3d_fwd(x, k, s)
        g = torch.randn(y_ref.shape, generator=gen).to(dtype)
        gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
        xb = torch.empty(x.numel() + 1, dtype=dtype, device=DEV)
        xd = xb[1:].view(shape)
        xd.copy_(x.to(DEV))
        yb = torch.empty(y_ref.numel() + 1, dtype=dtype, device=DEV)
        yd = yb[1:].view(y_ref.shape)
        idx = torch.empty(y_ref.shape, dtype=torch.int64, device=DEV)
        mp.maxpool3d_fwd(xd, yd, idx, k, s)
        gb = torch.empty(g.numel() + 1, dtype=dtype, device=DEV)
        gd = gb[1:].view(g.shape)
        gd.copy_(g.to(DEV))
        ginb = torch.empty(x.numel() + 1, dtype=dtype, device=DEV)
        gind = ginb[1:].view(shape)
        mp.maxpool3d_bwd(gd, idx, gind, k, s)
        torch.cuda.synchronize()
        assert torch.equal(idx.cpu(), i_ref)
        assert_bits_equal(yd.cpu(), y_ref, "y (unaligned)")
        assert_bits_equal(gind.cpu(), gin_ref, "grad_in (unaligned)")


@pytest.mark.parametrize("dtype", (torch.float16, torch.bfloat16), ids=str)
@pytest.mark.parametrize("window", [((2, 2, 2), (2, 2, 2)), ((3, 3, 3), (2, 2, 2))], ids=["k2s2", "k3s2"])
def test_stride2_forward_unaligned_outputs(window, dtype):
    # Aligned input, y and idx one element past a 16-byte boundary: the
    # stride-2 kernels copy their outputs element by element.
    k, s = window
    shape = (2, 3, 10, 22, 48)
    gen = torch.Generator().manual_seed(32)
    x = random_input(gen, shape, dtype, "ties")
    y_ref, i_ref = oracle.maxpool3d_fwd(x, k, s)
    assert mp.maxpool3d_fwd_plan(shape, k, s, dtype) == "fwd_s2"
    yb = torch.empty(y_ref.numel() + 1, dtype=dtype, device=DEV)
    ib = torch.empty(y_ref.numel() + 1, dtype=torch.int64, device=DEV)
    yd, idd = yb[1:].view(y_ref.shape), ib[1:].view(y_ref.shape)
    mp.maxpool3d_fwd(x.to(DEV), yd, idd, k, s)
    torch.cuda.synchronize()
    assert torch.equal(idd.cpu(), i_ref)
    assert_bits_equal(yd.cpu(), y_ref, "y (unaligned outputs)")


@pytest.mark.parametrize("algo", [mp.BWD_AUTO, mp.BWD_ATOMIC])
def test_guard_bands_untouched(algo):
    # Outputs live inside larger buffers filled with a sentinel; nothing
    # outside the output ranges may change.
    gen = torch.Generator().manual_seed(41)
    for dtype in DTYPES:
        for k, s, shape in (FIXED_CASES[0], FIXED_CASES[1], FIXED_CASES[6]):
            x = random_input(gen, shape, dtype, "normal").to(DEV)
            out = mp.pool_out_size(shape[2:], k, s)
            oshape = shape[:2] + out
            no, ni = 1, 1
            for v in oshape:
                no *= v
            for v in shape:
                ni *= v
            pad = 64
            yb = torch.full((no + 2 * pad,), 7.0, dtype=dtype, device=DEV)
            ib = torch.full((no + 2 * pad,), -7, dtype=torch.int64, device=DEV)
            gb = torch.full((ni + 2 * pad,), 5.0, dtype=dtype, device=DEV)
            y, idx, gin = yb[pad:pad + no].view(oshape), ib[pad:pad + no].view(oshape), \
                gb[pad:pad + ni].view(shape)
            mp.maxpool3d_fwd(x, y, idx, k, s)
            g = torch.randn(oshape, generator=gen).to(dtype).to(DEV)
            nbytes = mp.maxpool3d_bwd_workspace_bytes(shape, dtype, algo)
            ws = torch.empty(nbytes // 4, dtype=torch.float32, device=DEV) if nbytes else None
            mp.maxpool3d_bwd(g, idx, gin, k, s, algo=algo, workspace=ws)
            torch.cuda.synchronize()
            for buf, val in ((yb, 7.0), (ib, -7), (gb, 5.0)):
                assert bool((buf[:pad] == val).all()) and bool((buf[-pad:] == val).all())


def test_large_plane_offsets():
    # In-plane offsets above 2^24 (not exact in binary32) must stay exact.
    shape = (1, 1, 64, 512, 1024)
    gen = torch.Generator().manual_seed(51)
    x = torch.randn(shape, generator=gen).to(torch.bfloat16)
    for k, s in (((2, 2, 2), (2, 2, 2)), ((3, 3, 3), (2, 2, 2))):
        y_ref, i_ref = oracle.maxpool3d_fwd(x, k, s)
        y, idx = gpu_fwd(x, kernel=k, stride=s)
        assert torch.equal(idx, i_ref)
        assert_bits_equal(y, y_ref, "y")
        g = torch.randn(y_ref.shape, generator=gen).to(torch.bfloat16)
        assert_bits_equal(gpu_bwd(g, i_ref, shape, k, s), oracle.maxpool3d_bwd(g, i_ref, shape[2:]),
                          "grad_in")


# Shapes aimed at the stride-2 forward kernel (16-bit types, rows a multiple
# of 8 elements): tails in OH (tiles of 4 rows) and OW (chunks of 4 outputs),
# depths that split into several groups, and NaN/Inf (exact fallback).
S2_SHAPES = [(1, 3, 2, 2, 8), (2, 2, 3, 5, 16), (1, 2, 7, 9, 24), (1, 1, 5, 17, 40),
             (2, 3, 16, 34, 112), (1, 2, 33, 6, 64), (3, 1, 4, 11, 8)]


@pytest.mark.parametrize("dtype", (torch.float16, torch.bfloat16), ids=str)
@pytest.mark.parametrize("window", [((2, 2, 2), (2, 2, 2)), ((3, 3, 3), (2, 2, 2))], ids=["k2s2", "k3s2"])
@pytest.mark.parametrize("shape", S2_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("kind", KINDS)
def test_stride2_forward(shape, window, dtype, kind):
    k, s = window
    if any(i < kk for i, kk in zip(shape[2:], k)):
        pytest.skip("window larger than input")
    assert mp.maxpool3d_fwd_plan(shape, k, s, dtype) == "fwd_s2"
    gen = torch.Generator().manual_seed(5000 + 97 * S2_SHAPES.index(shape) + 7 * k[0] + KINDS.index(kind))
    x = random_input(gen, shape, dtype, kind)
    y_ref, i_ref = oracle.maxpool3d_fwd(x, k, s)
    y, idx = gpu_fwd(x, kernel=k, stride=s)
    assert torch.equal(idx, i_ref), f"idx differs ({shape}, {k}, {kind})"
    assert_bits_equal(y, y_ref, "y")


@pytest.mark.parametrize("dtype", (torch.float16, torch.bfloat16), ids=str)
def test_stride2_forward_subnormals_and_signed_zeros(dtype):
    gen = torch.Generator().manual_seed(61)
    shape = (2, 2, 5, 9, 32)
    tiny = torch.finfo(dtype).smallest_normal
    x = (torch.randint(-4, 5, shape, generator=gen).float() * tiny / 8).to(dtype)
    for k, s in (((2, 2, 2), (2, 2, 2)), ((3, 3, 3), (2, 2, 2))):
        y_ref, i_ref = oracle.maxpool3d_fwd(x, k, s)
        y, idx = gpu_fwd(x, kernel=k, stride=s)
        assert torch.equal(idx, i_ref)
        assert_bits_equal(y, y_ref, "y")


DISJOINT_CASES = [((2, 2, 2), (2, 2, 2), (2, 3, 6, 10, 64)), ((1, 2, 1), (3, 2, 4), (2, 2, 7, 9, 32)),
                  ((1, 1, 1), (1, 1, 1), (1, 2, 3, 4, 16)), ((2, 1, 3), (2, 3, 8), (1, 3, 9, 5, 48)),
                  ((3, 3, 2), (3, 3, 2), (2, 2, 9, 12, 8))]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(DISJOINT_CASES)))
def test_disjoint_backward_row_chunks(case, dtype):
    k, s, shape = DISJOINT_CASES[case]
    assert mp.maxpool3d_bwd_plan(shape, mp.pool_out_size(shape[2:], k, s), k, s, dtype) == "bwd_disjoint"
    gen = torch.Generator().manual_seed(7000 + case)
    x = random_input(gen, shape, dtype, "ties")
    _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    g = torch.randn(i_ref.shape, generator=gen).to(dtype)
    assert_bits_equal(gpu_bwd(g, i_ref, shape, k, s), oracle.maxpool3d_bwd(g, i_ref, shape[2:]),
                      "grad_in")


def test_no_device_error_flags_after_suite():
    # The forward's copy pipeline never timed out during these tests.
    assert mp.mp3d_device_error_flags(clear=True) == 0


# Overlapping shapes with at most two windows over any position on every
# axis: the rolling ordered scatter. Several h-tiles per plane for the large
# planes, ragged rows (H*W not a multiple of the vector width), inputs
# claimed by up to eight windows, ties (many shared winners).
ROLL_CASES = [((3, 3, 3), (2, 2, 2), (2, 3, 40, 30, 24)), ((2, 2, 2), (1, 1, 1), (1, 2, 20, 33, 17)),
              ((3, 2, 3), (2, 1, 2), (2, 2, 13, 9, 40)), ((4, 4, 4), (3, 3, 3), (1, 2, 22, 19, 31)),
              ((3, 3, 3), (2, 2, 2), (1, 2, 24, 112, 112)), ((3, 3, 3), (2, 2, 2), (1, 2, 20, 113, 114)),
              ((2, 2, 2), (1, 1, 1), (1, 2, 12, 20, 16)), ((3, 3, 3), (2, 2, 2), (2, 2, 17, 31, 40)),
              # kernel < stride on d (uncovered slices), overlap on h and w
              ((1, 3, 2), (3, 2, 1), (2, 2, 10, 21, 30)),
              # a tall plane: many h-tiles
              ((3, 3, 3), (2, 2, 2), (1, 2, 7, 301, 45)),
              # wide rows: h-tiles of about 500 and 900 windows (two and four
              # windows per thread)
              ((3, 3, 3), (2, 2, 2), (1, 2, 9, 64, 200)), ((3, 3, 3), (2, 2, 2), (1, 2, 5, 20, 600))]
# Adaptive shapes with at most two windows over any position.
ROLL_ADAPTIVE = [((2, 3, 30, 50, 50), (8, 12, 12)), ((1, 2, 10, 12, 9), (4, 5, 4)),
                 ((2, 2, 9, 7, 13), (5, 4, 8)), ((1, 3, 5, 6, 7), (3, 3, 3)),
                 ((1, 2, 33, 250, 17), (10, 60, 5))]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(ROLL_CASES)))
def test_overlap_roll_backward(case, dtype):
    k, s, shape = ROLL_CASES[case]
    out = mp.pool_out_size(shape[2:], k, s)
    assert mp.maxpool3d_bwd_plan(shape, out, k, s, dtype) == "bwd_overlap_roll"
    gen = torch.Generator().manual_seed(8000 + case)
    x = random_input(gen, shape, dtype, "ties")
    _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    g = torch.randn(i_ref.shape, generator=gen).to(dtype)
    assert_bits_equal(gpu_bwd(g, i_ref, shape, k, s), oracle.maxpool3d_bwd(g, i_ref, shape[2:]),
                      "grad_in")


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(ROLL_ADAPTIVE)))
def test_overlap_roll_backward_adaptive(case, dtype):
    shape, out = ROLL_ADAPTIVE[case]
    assert mp.maxpool3d_bwd_plan(shape, out, None, None, dtype) == "bwd_overlap_roll"
    gen = torch.Generator().manual_seed(8050 + case)
    x = random_input(gen, shape, dtype, "ties")
    _, i_ref = oracle.adaptive_maxpool3d_fwd(x, out)
    g = torch.randn(i_ref.shape, generator=gen).to(dtype)
    assert_bits_equal(gpu_bwd(g, i_ref, shape), oracle.maxpool3d_bwd(g, i_ref, shape[2:]),
                      "grad_in")


# The same overlapping shapes with grad_in one element past a 16-byte
# boundary: the rolling scatter needs aligned rows, so the tiled owner gather
# (and, for its compiled windows, the chunk gather) takes them. Plus shapes
# with three windows over a position along one axis, which the tiled gather
# takes at any alignment.
TILE_ONLY = [((3, 2, 2), (1, 2, 2), (2, 2, 15, 18, 20)), ((2, 4, 3), (2, 1, 2), (1, 3, 9, 20, 33))]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(ROLL_CASES) + len(TILE_ONLY)))
def test_overlap_tile_backward(case, dtype):
    allc = ROLL_CASES + TILE_ONLY
    k, s, shape = allc[case]
    out = mp.pool_out_size(shape[2:], k, s)
    offset = 1 if case < len(ROLL_CASES) else 0
    if offset == 0:
        assert mp.maxpool3d_bwd_plan(shape, out, k, s, dtype) == "bwd_overlap_tile"
    gen = torch.Generator().manual_seed(8200 + case)
    x = random_input(gen, shape, dtype, "ties")
    _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    g = torch.randn(i_ref.shape, generator=gen).to(dtype)
    assert_bits_equal(gpu_bwd(g, i_ref, shape, k, s, offset=offset),
                      oracle.maxpool3d_bwd(g, i_ref, shape[2:]), "grad_in")


# Gradients holding -0 and +0 on inputs claimed by several windows: a sum
# whose terms are all -0 is -0, any other all-zero sum is +0, and inputs no
# window chose are +0. Also infinite and NaN gradients. Run on the rolling
# scatter (aligned grad_in) and on the gathers (offset grad_in).
@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("window", [((3, 3, 3), (2, 2, 2)), ((2, 2, 2), (1, 1, 1))], ids=["k3s2", "k2s1"])
@pytest.mark.parametrize("grad", ["mixed_zeros", "all_negative_zero", "non_finite"])
@pytest.mark.parametrize("offset", [0, 1], ids=["roll", "gather"])
def test_overlap_backward_signed_zero_gradients(window, dtype, grad, offset):
    k, s = window
    shape = (2, 2, 11, 14, 24)
    out = mp.pool_out_size(shape[2:], k, s)
    assert mp.maxpool3d_bwd_plan(shape, out, k, s, dtype) == "bwd_overlap_roll"
    gen = torch.Generator().manual_seed(8100)
    x = random_input(gen, shape, dtype, "ties")
    _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    if grad == "all_negative_zero":
        g = torch.full(i_ref.shape, -0.0).to(dtype)
    elif grad == "non_finite":
        # +-inf and NaN gradients (plus one -0): sums through them follow
        # IEEE rules in the same order as the oracle
        r = torch.rand(i_ref.shape, generator=gen)
        g = torch.randint(-2, 3, i_ref.shape, generator=gen).float()
        g = torch.where(r < 0.02, torch.tensor(float("inf")), g)
        g = torch.where((r >= 0.02) & (r < 0.04), torch.tensor(float("-inf")), g)
        g = torch.where((r >= 0.04) & (r < 0.05), torch.tensor(float("nan")), g)
        g.view(-1)[0] = -0.0
        g = g.to(dtype)
    else:
        r = torch.rand(i_ref.shape, generator=gen)
        g = torch.where(r < 0.4, torch.tensor(-0.0), torch.where(r < 0.7, torch.tensor(0.0),
                                                                 torch.randint(-2, 3, i_ref.shape,
                                                                               generator=gen).float()))
        g = g.to(dtype)
    ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    if grad != "non_finite":
        assert bool((bits(ref) == bits(torch.tensor(-0.0).to(dtype))).any())
    assert_bits_equal(gpu_bwd(g, i_ref, shape, k, s, offset=offset), ref, "grad_in")


# The same gradients on wide rows (about 900 windows per h-tile, the
# specialised 3x3x3 stride-2 form with 16-byte aligned rows).
@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("grad", ["mixed_zeros", "all_negative_zero"])
def test_overlap_roll_signed_zero_gradients_wide_rows(dtype, grad):
    k, s = (3, 3, 3), (2, 2, 2)
    shape = (1, 2, 5, 20, 600)
    out = mp.pool_out_size(shape[2:], k, s)
    assert mp.maxpool3d_bwd_plan(shape, out, k, s, dtype) == "bwd_overlap_roll"
    gen = torch.Generator().manual_seed(8101)
    x = random_input(gen, shape, dtype, "ties")
    _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    if grad == "all_negative_zero":
        g = torch.full(i_ref.shape, -0.0).to(dtype)
    else:
        r = torch.rand(i_ref.shape, generator=gen)
        g = torch.where(r < 0.4, torch.tensor(-0.0), torch.where(r < 0.7, torch.tensor(0.0),
                                                                 torch.randint(-2, 3, i_ref.shape,
                                                                               generator=gen).float()))
        g = g.to(dtype)
    ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    assert bool((bits(ref) == bits(torch.tensor(-0.0).to(dtype))).any())
    assert_bits_equal(gpu_bwd(g, i_ref, shape, k, s), ref, "grad_in")


# Values-only forward (idx NULL): y is the same, bit for bit, on every
# forward path; no index buffer is touched.
VALUES_ONLY = [
    ("fwd_s2", (3, 3, 3), (2, 2, 2), None, (1, 2, 9, 20, 48), torch.float16),
    ("fwd_s2", (2, 2, 2), (2, 2, 2), None, (1, 2, 8, 6, 32), torch.bfloat16),    # 2x2x2 tiling
    ("fwd_s2", (2, 2, 2), (2, 2, 2), None, (1, 2, 9, 7, 32), torch.float16),
    ("fwd_s2", (3, 3, 3), (2, 2, 2), None, (2, 3, 11, 24, 64), torch.bfloat16),
    ("fwd_slab", None, None, (5, 4, 8), (2, 2, 9, 7, 13), torch.float32),
    ("fwd_roll", None, None, (8, 12, 12), (1, 3, 30, 50, 50), torch.float16),
    ("fwd_roll", None, None, (3, 4, 5), (2, 3, 7, 9, 13), torch.bfloat16),
    ("fwd_roll", None, None, (4, 20, 20), (1, 2, 9, 40, 40), torch.float16),      # bands of rows
    ("fwd_slab", None, None, (4, 20, 20), (1, 2, 9, 39, 41), torch.float16),      # keyed slab
    ("fwd_generic", (5, 5, 5), (3, 3, 3), None, (1, 1, 8, 120, 120), torch.float32),
    ("fwd_global", None, None, (1, 1, 1), (1, 3, 8, 14, 14), torch.float32),
]


@pytest.mark.parametrize("case", range(len(VALUES_ONLY)))
def test_values_only_forward(case):
    path, k, s, out, shape, dtype = VALUES_ONLY[case]
    gen = torch.Generator().manual_seed(9000 + case)
    x = random_input(gen, shape, dtype, "special")
    if k is not None:
        assert mp.maxpool3d_fwd_plan(shape, k, s, dtype) == path
        y_ref, _ = oracle.maxpool3d_fwd(x, k, s)
    else:
        assert mp.adaptive_maxpool3d_fwd_plan(shape, out, dtype) == path
        y_ref, _ = oracle.adaptive_maxpool3d_fwd(x, out)
    y = torch.empty(y_ref.shape, dtype=dtype, device=DEV)
    if k is not None:
        mp.maxpool3d_fwd(x.to(DEV), y, None, k, s)
    else:
        mp.adaptive_maxpool3d_fwd(x.to(DEV), y, None, out)
    torch.cuda.synchronize()
    assert_bits_equal(y.cpu(), y_ref, "y (values only)")


# Padding, dilation and ceil mode: forward values and indices, the ordered
# backward bit for bit, and the atomic form within its tolerance.
PADDED_CASES = [
    ((3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), False, (2, 3, 9, 20, 33)),
    ((3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), True, (1, 2, 8, 17, 30)),
    ((2, 2, 2), (2, 2, 2), (1, 1, 1), (1, 1, 1), False, (1, 3, 7, 11, 16)),
    ((3, 2, 3), (1, 2, 2), (1, 0, 1), (2, 1, 2), False, (1, 2, 9, 12, 21)),
    ((2, 3, 2), (2, 1, 3), (0, 1, 1), (3, 2, 1), True, (2, 2, 10, 9, 23)),
    ((2, 2, 2), (2, 2, 2), (0, 0, 0), (1, 1, 1), True, (1, 2, 9, 9, 9)),       # ceil adds a window
    ((4, 4, 4), (3, 3, 3), (2, 2, 2), (1, 1, 1), True, (1, 2, 11, 14, 19)),
    ((3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), False, (1, 2, 6, 112, 112)),  # wide planes
    ((3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), False, (1, 3, 8, 56, 56)),    # bands of output rows
    ((2, 2, 2), (2, 2, 2), (0, 0, 0), (1, 1, 1), True, (1, 3, 8, 9, 10)),      # ceil mode, clipped
    ((3, 3, 3), (1, 2, 2), (1, 1, 1), (1, 1, 1), True, (2, 1, 8, 40, 24)),     # depth stride 1 (3 covers)
]


def _padded_fwd_path(shape, k, s, p, dl, cm, dtype):
    """The forward path the library takes for a padded geometry: the stride-2
    kernel for 16-bit 3x3x3 stride-2 windows with padding <= 1, rows a
    multiple of 8 elements and floor sizes; else, for 16-bit types with
    dilation 1 and plane volumes a multiple of 8, the depth walk (clipped
    windows); else the thread-per-output kernel."""
    floor = all(o == (i + 2 * pp - kk) // ss + 1 for o, i, kk, ss, pp in
                zip(mp.pool_out_size_ex(shape[2:], k, s, p, dl, cm), shape[2:], k, s, p))
    if (dtype != torch.float32 and tuple(k) == (3, 3, 3) and tuple(s) == (2, 2, 2) and
            tuple(dl) == (1, 1, 1) and max(p) <= 1 and shape[4] % 8 == 0 and shape[4] <= 1024 and floor):
        return "fwd_s2"
    if (dtype != torch.float32 and tuple(dl) == (1, 1, 1) and k[0] <= 2 * s[0] and
            (shape[2] * shape[3] * shape[4]) % 8 == 0):
        return "fwd_roll"
    return "fwd_padded"


def _gpu_fwd_ex(x_cpu, k, s, p, dl, cm):
    x = x_cpu.to(DEV)
    out = mp.pool_out_size_ex(x.shape[2:], k, s, p, dl, cm)
    y = torch.empty(x.shape[:2] + out, dtype=x.dtype, device=DEV)
    idx = torch.empty(x.shape[:2] + out, dtype=torch.int64, device=DEV)
    mp.maxpool3d_fwd_ex(x, y, idx, k, s, p, dl, cm)
    torch.cuda.synchronize()
    return y.cpu(), idx.cpu()


def _gpu_bwd_ex(g_cpu, idx_cpu, in_shape, k, s, p, dl, cm, algo=mp.BWD_AUTO):
    g, idx = g_cpu.to(DEV), idx_cpu.to(DEV)
    gin = torch.empty(in_shape, dtype=g.dtype, device=DEV)
    nbytes = mp.maxpool3d_bwd_workspace_bytes(in_shape, g.dtype, algo)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=DEV) if nbytes else None
    mp.maxpool3d_bwd_ex(g, idx, gin, k, s, p, dl, cm, algo=algo, workspace=ws)
    torch.cuda.synchronize()
    return gin.cpu()


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(PADDED_CASES)))
def test_padded_fwd_bwd(case, dtype):
    k, s, p, dl, cm, shape = PADDED_CASES[case]
    # 16-bit types with dilation 1 and plane volumes a multiple of 8 take the
    # depth walk (clipped windows); the rest the thread-per-output kernel
    assert mp.maxpool3d_fwd_ex_plan(shape, k, s, p, dl, cm, dtype) == _padded_fwd_path(shape, k, s, p, dl, cm,
                                                                                     dtype)
    gen = torch.Generator().manual_seed(9500 + case)
    x = random_input(gen, shape, dtype, KINDS[case % 3])
    y_ref, i_ref = oracle.maxpool3d_fwd_ex(x, k, s, p, dl, cm)
    y, idx = _gpu_fwd_ex(x, k, s, p, dl, cm)
    assert torch.equal(idx, i_ref)
    assert_bits_equal(y, y_ref, "y (padded)")
    g = torch.randn(y_ref.shape, generator=gen).to(dtype)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    # undilated windows take the rolling ordered scatter, dilated ones the
    # direct gather; both are bit-exact
    two_cover = all(kk <= 2 * ss for kk, ss in zip(k, s))
    want = "bwd_overlap_roll" if dl == (1, 1, 1) and two_cover else "bwd_padded"
    assert mp.maxpool3d_bwd_ex_plan(shape, y_ref.shape[2:], k, s, p, dl, cm, dtype) == want
    assert_bits_equal(_gpu_bwd_ex(g, i_ref, shape, k, s, p, dl, cm), gin_ref, "grad_in (padded)")
    gin_a = _gpu_bwd_ex(g, i_ref, shape, k, s, p, dl, cm, algo=mp.BWD_ATOMIC)
    assert _atomic_tolerance_ok(gin_a, gin_ref, g, i_ref, dtype)


PADDED_S2_CASES = [
    ((1, 1, 1), (2, 3, 16, 56, 56)),      # even sizes, the bench's padded geometry
    ((1, 1, 1), (1, 2, 9, 23, 112)),      # odd D and H: the last windows clipped below
    ((0, 1, 1), (1, 3, 8, 30, 112)),
    ((1, 0, 1), (1, 2, 7, 17, 112)),
    ((1, 1, 0), (2, 1, 10, 15, 112)),
    ((0, 0, 1), (1, 2, 5, 9, 8)),         # one chunk per row: the left edge everywhere
    ((1, 0, 0), (1, 2, 6, 11, 112)),
    ((1, 1, 1), (1, 2, 5, 112, 112)),     # several bands of output rows
]
# (rows of 112 elements give the backward's h-tiles more than 256 windows,
# which the compiled 3x3x3 rolling form takes)


@pytest.mark.parametrize("dtype", (torch.float16, torch.bfloat16), ids=str)
@pytest.mark.parametrize("case", range(len(PADDED_S2_CASES)))
def test_padded_stride2_forward(case, dtype):
    # 3x3x3 windows, stride 2, padding <= 1: the stride-2 kernel with clamped
    # slices, rows and columns; ties, signed zeros, infinities and NaNs; then
    # the backward of the same windows
    p, shape = PADDED_S2_CASES[case]
    k, s = (3, 3, 3), (2, 2, 2)
    assert mp.maxpool3d_fwd_ex_plan(shape, k, s, p, (1, 1, 1), False, dtype) == "fwd_s2"
    gen = torch.Generator().manual_seed(9700 + case)
    for kind in ("ties", "special", "normal"):
        x = random_input(gen, shape, dtype, kind)
        y_ref, i_ref = oracle.maxpool3d_fwd_ex(x, k, s, p, (1, 1, 1), False)
        y, idx = _gpu_fwd_ex(x, k, s, p, (1, 1, 1), False)
        assert torch.equal(idx, i_ref), kind
        assert_bits_equal(y, y_ref, f"y (padded stride 2, {kind})")
    # values only, and outputs one element past a 16-byte boundary
    xd = x.to(DEV)
    yv = torch.empty(y_ref.shape, dtype=dtype, device=DEV)
    mp.maxpool3d_fwd_ex(xd, yv, None, k, s, p)
    yb = torch.empty(y_ref.numel() + 1, dtype=dtype, device=DEV)
    ib = torch.empty(y_ref.numel() + 1, dtype=torch.int64, device=DEV)
    yu, iu = yb[1:].view(y_ref.shape), ib[1:].view(y_ref.shape)
    mp.maxpool3d_fwd_ex(xd, yu, iu, k, s, p)
    torch.cuda.synchronize()
    assert_bits_equal(yv.cpu(), y_ref, "y (padded stride 2, values only)")
    assert_bits_equal(yu.cpu(), y_ref, "y (padded stride 2, unaligned)")
    assert torch.equal(iu.cpu(), i_ref)
    # the backward of the same padded windows (the compiled 3x3x3 form where
    # rows and planes are 16-byte multiples), -0 gradients mixed in
    g = torch.randn(y_ref.shape, generator=gen)
    g = torch.where(torch.rand(y_ref.shape, generator=gen) < 0.1, torch.tensor(-0.0), g).to(dtype)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    assert mp.maxpool3d_bwd_ex_plan(shape, y_ref.shape[2:], k, s, p, (1, 1, 1), False, dtype) == "bwd_overlap_roll"
    assert_bits_equal(_gpu_bwd_ex(g, i_ref, shape, k, s, p, (1, 1, 1), False), gin_ref,
                      "grad_in (padded stride 2)")
    gin_a = _gpu_bwd_ex(g, i_ref, shape, k, s, p, (1, 1, 1), False, algo=mp.BWD_ATOMIC)
    assert _atomic_tolerance_ok(gin_a, gin_ref, g, i_ref, dtype)


def test_padded_plain_geometry_matches_plain_entry_points():
    # no padding, no dilation, floor sizes: the same paths and results
    gen = torch.Generator().manual_seed(9600)
    shape, k, s = (1, 2, 16, 40, 48), (3, 3, 3), (2, 2, 2)
    x = random_input(gen, shape, torch.float16, "ties")
    y0, i0 = gpu_fwd(x, kernel=k, stride=s)
    y1, i1 = _gpu_fwd_ex(x, k, s, (0, 0, 0), (1, 1, 1), False)
    assert torch.equal(i0, i1)
    assert_bits_equal(y0, y1, "y")
    g = torch.randn(y0.shape, generator=gen).half()
    assert_bits_equal(gpu_bwd(g, i0, shape, k, s), _gpu_bwd_ex(g, i0, shape, k, s, (0, 0, 0), (1, 1, 1),
                                                             False), "grad_in")


# Backward without stored indices: the same bits as the backward through
# the forward's indices (oracle forward, then oracle backward).
RECOMPUTE_CASES = [
    ((2, 2, 2), (2, 2, 2), None, (2, 3, 8, 12, 64)),        # 2x2x2 tiling, fused kernel
    ((2, 2, 2), (2, 2, 2), None, (1, 2, 9, 11, 40)),        # not a tiling
    ((3, 3, 3), (2, 2, 2), None, (1, 2, 9, 13, 21)),        # overlapping
    ((1, 3, 2), (3, 2, 1), None, (1, 2, 10, 9, 14)),
    (None, None, (3, 4, 5), (1, 2, 9, 12, 15)),             # adaptive, divisible
    (None, None, (4, 5, 6), (2, 2, 10, 11, 13)),            # adaptive, overlapping
]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(RECOMPUTE_CASES)))
def test_backward_recompute(case, dtype):
    k, s, out, shape = RECOMPUTE_CASES[case]
    gen = torch.Generator().manual_seed(9700 + case)
    x = random_input(gen, shape, dtype, KINDS[case % 3])
    if k is not None:
        _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    else:
        _, i_ref = oracle.adaptive_maxpool3d_fwd(x, out)
    g = torch.randn(i_ref.shape, generator=gen).to(dtype)
    ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
    want = "bwd_recompute_k2s2" if case == 0 else "bwd_recompute_direct"
    assert mp.maxpool3d_bwd_recompute_plan(shape, i_ref.shape[2:], k, s, dtype) == want
    gin = torch.empty(shape, dtype=dtype, device=DEV)
    mp.maxpool3d_bwd_recompute(x.to(DEV), g.to(DEV), gin, k, s)
    torch.cuda.synchronize()
    assert_bits_equal(gin.cpu(), ref, "grad_in (recomputed argmax)")


# Channels-last layout: the NCDHW results (oracle) with the channel axis
# moved last; 16-byte chunks across channels when C allows, element access
# otherwise (odd C, or buffers one element off a 16-byte boundary).
NDHWC_CASES = [
    ((3, 3, 3), (2, 2, 2), None, (2, 9, 13, 11, 16)),
    ((2, 2, 2), (2, 2, 2), None, (1, 8, 10, 12, 24)),
    ((2, 3, 2), (1, 2, 3), None, (2, 7, 9, 10, 5)),         # odd channel count
    (None, None, (4, 5, 3), (1, 10, 11, 9, 8)),             # adaptive, overlapping
    (None, None, (1, 1, 1), (2, 4, 6, 5, 32)),              # global
    ((3, 3, 3), (2, 2, 2), None, (1, 7, 9, 11, 16)),        # packed 16-bit form, special values
    ((2, 2, 2), (2, 2, 2), None, (2, 6, 8, 10, 24)),
    ((3, 2, 3), (2, 2, 1), None, (1, 8, 7, 9, 32)),
    (None, None, (3, 4, 5), (2, 6, 9, 10, 8)),              # adaptive, special values
    ((3, 3, 3), (2, 1, 1), None, (1, 7, 8, 9, 16)),         # depth walk, stride 1 in (h, w)
    ((3, 3, 3), (2, 3, 3), None, (2, 9, 10, 11, 24)),       # depth walk, disjoint in (h, w)
]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(NDHWC_CASES)))
@pytest.mark.parametrize("offset", [0, 1], ids=["aligned", "offset"])
def test_channels_last(case, dtype, offset):
    k, s, out, shape = NDHWC_CASES[case]
    gen = torch.Generator().manual_seed(9800 + case)
    x = random_input(gen, shape, dtype, KINDS[case % 3])          # (N, D, H, W, C)
    xc = x.permute(0, 4, 1, 2, 3).contiguous()                    # (N, C, D, H, W)
    if k is not None:
        y_ref, i_ref = oracle.maxpool3d_fwd(xc, k, s)
    else:
        y_ref, i_ref = oracle.adaptive_maxpool3d_fwd(xc, out)
    oshape = (shape[0],) + tuple(y_ref.shape[2:]) + (shape[4],)

    def buf(shp, dt):
        n = 1
        for v in shp:
            n *= v
        return torch.empty(n + offset, dtype=dt, device=DEV)[offset:].view(shp)

    xd = buf(shape, dtype)
    xd.copy_(x.to(DEV))
    y, idx = buf(oshape, dtype), buf(oshape, torch.int64)
    if k is not None:
        mp.maxpool3d_fwd_ndhwc(xd, y, idx, k, s)
    else:
        mp.adaptive_maxpool3d_fwd_ndhwc(xd, y, idx, out)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), i_ref.permute(0, 2, 3, 4, 1))
    assert_bits_equal(y.cpu(), y_ref.permute(0, 2, 3, 4, 1).contiguous(), "y (channels last)")
    g = torch.randn(y_ref.shape, generator=gen).to(dtype)         # (N, C, OD, OH, OW)
    if case % 2:
        # signed zeros and small integers: sums of lone -0 terms stay -0,
        # -0 + +0 is +0, cancellations give +0
        pick = torch.randint(0, 5, y_ref.shape, generator=gen)
        g = torch.tensor([-0.0, 0.0, -0.0, 1.0, -1.0])[pick].to(dtype)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[1:4])
    gd = buf(oshape, dtype)
    gd.copy_(g.permute(0, 2, 3, 4, 1).to(DEV))
    gin = buf(shape, dtype)
    mp.maxpool3d_bwd_ndhwc(gd, idx, gin, k, s)
    torch.cuda.synchronize()
    assert_bits_equal(gin.cpu(), gin_ref.permute(0, 2, 3, 4, 1).contiguous(), "grad_in (channels last)")


# The channels-last rolling backward: tiles of input rows and columns per
# CTA (several per axis here, with ragged last tiles), several channel
# groups, windows with two covers per axis (stride 1 included), adaptive
# windows, a ring as deep as the input (global windows), integer inputs with
# many ties (windows sharing their chosen input) and signed-zero gradients.
NDHWC_ROLL_CASES = [
    ((3, 3, 3), (2, 2, 2), None, (2, 9, 30, 29, 16)),
    ((3, 3, 3), (2, 2, 2), None, (1, 8, 17, 35, 40)),
    ((2, 2, 2), (1, 1, 1), None, (1, 6, 20, 18, 8)),
    ((3, 2, 3), (2, 1, 2), None, (2, 7, 16, 19, 24)),
    ((3, 3, 2), (2, 2, 2), None, (2, 8, 30, 30, 16)),       # disjoint along w
    ((2, 1, 2), (1, 1, 1), None, (1, 3, 5, 7, 8)),          # one-element along h
    (None, None, (4, 11, 10), (1, 10, 30, 29, 16)),
    (None, None, (3, 7, 9), (2, 9, 20, 33, 8)),
    (None, None, (1, 1, 1), (2, 4, 6, 5, 16)),
    ((3, 3, 3), (2, 2, 2), None, (1, 3, 3, 3, 128)),
]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(NDHWC_ROLL_CASES)))
def test_channels_last_rolling_backward(case, dtype):
    k, s, out, shape = NDHWC_ROLL_CASES[case]
    N, D, H, W, C = shape
    gen = torch.Generator().manual_seed(9900 + case)
    x = torch.randint(-3, 4, (N, C, D, H, W), generator=gen).to(dtype)     # ties everywhere
    if k is not None:
        _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    else:
        _, i_ref = oracle.adaptive_maxpool3d_fwd(x, out)
    osz = tuple(i_ref.shape[2:])
    if case % 2:
        pick = torch.randint(0, 5, i_ref.shape, generator=gen)
        g = torch.tensor([-0.0, 0.0, -0.0, 1.0, -1.5])[pick].to(dtype)
    else:
        g = torch.randn(i_ref.shape, generator=gen).to(dtype)
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, (D, H, W))
    assert mp.maxpool3d_bwd_ndhwc_plan((N, C, D, H, W), osz, k, s, dtype) == "bwd_ndhwc_roll"
    gd = g.permute(0, 2, 3, 4, 1).contiguous().to(DEV)
    idx = i_ref.permute(0, 2, 3, 4, 1).contiguous().to(DEV)
    gin = torch.full(shape, float("nan"), dtype=dtype, device=DEV)
    mp.maxpool3d_bwd_ndhwc(gd, idx, gin, k, s)
    torch.cuda.synchronize()
    assert_bits_equal(gin.cpu(), gin_ref.permute(0, 2, 3, 4, 1).contiguous(),
                      "grad_in (channels-last rolling backward)")


# binary32 channel counts that hold 16 but not 32 bytes of channels: groups
# of four channels per CTA (half-sector stores)
@pytest.mark.parametrize("case", [((3, 3, 3), (2, 2, 2), (1, 8, 17, 35, 12)),
                                  ((2, 2, 2), (1, 1, 1), (2, 5, 9, 11, 4))], ids=["k3s2_c12", "k2s1_c4"])
def test_channels_last_rolling_backward_groups_of_four(case):
    k, s, shape = case
    N, D, H, W, C = shape
    gen = torch.Generator().manual_seed(9950 + C)
    x = torch.randint(-3, 4, (N, C, D, H, W), generator=gen).to(torch.float32)
    _, i_ref = oracle.maxpool3d_fwd(x, k, s)
    pick = torch.randint(0, 5, i_ref.shape, generator=gen)
    g = torch.tensor([-0.0, 0.0, -0.0, 1.0, -1.5])[pick]
    gin_ref = oracle.maxpool3d_bwd(g, i_ref, (D, H, W))
    assert mp.maxpool3d_bwd_ndhwc_plan((N, C, D, H, W), tuple(i_ref.shape[2:]), k, s,
                                       torch.float32) == "bwd_ndhwc_roll"
    gin = torch.full(shape, float("nan"), device=DEV)
    mp.maxpool3d_bwd_ndhwc(g.permute(0, 2, 3, 4, 1).contiguous().to(DEV),
                           i_ref.permute(0, 2, 3, 4, 1).contiguous().to(DEV), gin, k, s)
    torch.cuda.synchronize()
    assert_bits_equal(gin.cpu(), gin_ref.permute(0, 2, 3, 4, 1).contiguous(), "grad_in (groups of four)")


# The slab and rolling forwards for 16-bit types rank elements by one
# unsigned word (value order key, then earliest offset). Arbitrary bit patterns pin that
# order against the scan's rule: NaNs of either sign and any payload (the
# first NaN wins), +0 against -0 (the first wins), subnormals, +-inf. Slab
# starts off a 16-byte boundary take the element-wise head and tail.
ANY_BITS_CASES = [
    ((2, 3, 30, 50, 50), (8, 12, 12)),
    ((2, 3, 7, 9, 13), (3, 4, 5)),
    ((1, 2, 5, 3, 3), (5, 3, 3)),       # one-element windows
    ((3, 1, 6, 6, 6), (1, 1, 1)),       # one window over a whole plane
    ((1, 2, 9, 40, 40), (4, 20, 20)),   # more outputs per depth than one CTA's threads (bands)
    ((1, 2, 9, 39, 41), (4, 20, 20)),   # the same, odd plane volume (keyed slab)
    ((2, 2, 7, 5, 9), (8, 6, 4)),       # more depth windows than slices
    ((1, 3, 8, 10, 12), (3, 4, 5)),     # plane pairs (volume a multiple of 8), a lone last plane
    ((1, 5, 16, 8, 8), (6, 3, 3)),
    ((1, 3, 8, 4, 10), (9, 3, 5)),      # plane pairs, more depth windows than slices
    ((1, 2, 6, 96, 64), (3, 40, 30)),   # plane pairs in bands of output rows (1200 outputs a depth)
]


def _any_bits(gen, shape, dtype, nan_share):
    b = torch.randint(0, 1 << 16, shape, generator=gen, dtype=torch.int32)
    if nan_share:
        exp_bits = 0x7C00 if dtype == torch.float16 else 0x7F80
        mant = (~exp_bits) & 0x7FFF
        nan = (torch.randint(0, 2, shape, generator=gen, dtype=torch.int32) << 15) | exp_bits | \
            (torch.randint(1, mant + 1, shape, generator=gen, dtype=torch.int32))
        pick = torch.rand(shape, generator=gen) < nan_share
        b = torch.where(pick, nan, b)
    zeros = torch.rand(shape, generator=gen) < 0.15        # many +-0 ties
    b = torch.where(zeros, torch.randint(0, 2, shape, generator=gen, dtype=torch.int32) << 15, b)
    b = torch.where(b >= 1 << 15, b - (1 << 16), b)      # the same 16 bits as a signed value
    return b.to(torch.int16).view(dtype)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=str)
@pytest.mark.parametrize("nan_share", [0.0, 0.02, 0.5])
@pytest.mark.parametrize("case", range(len(ANY_BITS_CASES)))
def test_slab_forward_any_bits(case, nan_share, dtype):
    shape, out = ANY_BITS_CASES[case]
    assert mp.adaptive_maxpool3d_fwd_plan(shape, out, dtype) in ("fwd_roll", "fwd_slab", "fwd_global")
    gen = torch.Generator().manual_seed(9700 + 10 * case + int(100 * nan_share))
    x = _any_bits(gen, shape, dtype, nan_share)
    y_ref, i_ref = oracle.adaptive_maxpool3d_fwd(x, out)
    y, idx = gpu_fwd(x, out_size=out)
    assert torch.equal(idx, i_ref), f"idx differs ({shape} -> {out}, nan share {nan_share})"
    assert torch.equal(bits(y), bits(y_ref)), "y must be the chosen element's own bits"


# The depth walk needs x on a 16-byte boundary; a view one element off takes
# another forward path with the same results.
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=str)
def test_depth_walk_unaligned_input_falls_back(dtype):
    shape, out = (1, 4, 8, 10, 12), (3, 4, 5)
    gen = torch.Generator().manual_seed(9990)
    x = random_input(gen, shape, dtype, "special")
    y_ref, i_ref = oracle.adaptive_maxpool3d_fwd(x, out)
    n = x.numel()
    xd = torch.empty(n + 1, dtype=dtype, device=DEV)[1:].view(shape)
    xd.copy_(x.to(DEV))
    y = torch.empty(y_ref.shape, dtype=dtype, device=DEV)
    idx = torch.empty(y_ref.shape, dtype=torch.int64, device=DEV)
    mp.adaptive_maxpool3d_fwd(xd, y, idx, out)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), i_ref)
    assert_bits_equal(y.cpu(), y_ref, "y (unaligned x)")


XROLL_CASES = [
    ((2, 3, 13, 17, 19), (3, 4, 4)),      # 87 inputs per window
    ((1, 4, 30, 50, 50), (8, 12, 12)),    # the adaptive workload's windows
    ((1, 2, 9, 200, 30), (2, 50, 7)),     # several windows per thread, rows in h-tiles
    ((2, 2, 7, 33, 41), (2, 2, 2)),       # windows of length 4 and 5 along d
]


@pytest.mark.parametrize("dtype", DTYPES, ids=str)
@pytest.mark.parametrize("case", range(len(XROLL_CASES)))
def test_adaptive_exchange_backward(case, dtype):
    # adaptive windows with many inputs each: the backward writes zeros, then
    # takes each chosen input's sum from its accumulator; compared with the
    # oracle bit for bit, with -0 gradients mixed in (an input chosen only by
    # -0 gradients gets -0, one chosen by -0 and +0 gets +0)
    shape, out = XROLL_CASES[case]
    gen = torch.Generator().manual_seed(9900 + case)
    for kind in ("ties", "special"):
        x = random_input(gen, shape, dtype, kind)
        _, i_ref = oracle.adaptive_maxpool3d_fwd(x, out)
        g = torch.randn(i_ref.shape, generator=gen)
        r = torch.rand(i_ref.shape, generator=gen)
        g = torch.where(r < 0.2, torch.tensor(-0.0), g)
        g = torch.where((r >= 0.2) & (r < 0.25), torch.tensor(0.0), g).to(dtype)
        gin_ref = oracle.maxpool3d_bwd(g, i_ref, shape[2:])
        assert mp.maxpool3d_bwd_plan(shape, out, None, None, dtype) == "bwd_overlap_roll"
        gin = gpu_bwd(g, i_ref, shape)
        assert_bits_equal(gin, gin_ref, f"grad_in (adaptive exchange backward, {kind})")
