"""Checks that pin the oracle to facts other than itself.

Each check takes a loaded ``oracle.Oracle`` and raises AssertionError when
it disagrees with what the pages and the mathematics fix: stated sizes,
worked examples, library routines (numpy's binary16 conversion and argmax,
torch's bfloat16 conversion), exact rational arithmetic, invariants and
brute force on tiny inputs. The same battery runs against deliberately
broken builds of the oracle (test_oracle_mutants.py) to show that each
plausible mistake is caught by at least one check.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DTYPES = (torch.float32, torch.float16, torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a CPU tensor as unsigned integers."""
    t = t.contiguous()
    if t.element_size() == 4:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------- formats

def check_f16_decode(orc):
    allbits = np.arange(65536, dtype=np.uint16)
    ref = allbits.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_to_f32(int(b)) for b in allbits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f16_encode_cases():
    rng = np.random.default_rng(7)
    finite = np.arange(65536, dtype=np.uint16).view(np.float16)
    finite = finite[np.isfinite(finite)].astype(np.float32)
    # midpoints between neighbouring binary16 values: exact ties
    pos = np.sort(np.unique(np.abs(finite)))
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)
    rnd = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * s for s in (1e-7, 1e-5, 1e-3, 1, 100, 3e4)])
    edge = np.array([65504, 65519, 65519.996, 65520, 65536, 1e9, 2.0**-24, 2.0**-25,
                     2.0**-25 * 1.0000001, 2.0**-26, 2.0**-14, 2.0**-14 * (1 - 2.0**-12),
                     np.inf, -np.inf, 0.0, -0.0], dtype=np.float32)
    return np.concatenate([finite, mids, -mids, rnd, edge, -edge])


def check_f16_encode(orc):
    xs = _f16_encode_cases()
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16(float(v)) for v in xs], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"f32->f16 differs for {xs[bad[:5]]}: {got[bad[:5]]} vs {ref[bad[:5]]}"
    got_nan = orc.f32_to_f16(float("nan"))
    assert (got_nan & 0x7C00) == 0x7C00 and (got_nan & 0x3FF) != 0


def check_bf16_decode(orc):
    allbits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = allbits.view(torch.bfloat16).float().numpy()
    got = np.array([orc.bf16_to_f32(int(b) & 0xFFFF) for b in allbits.tolist()], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def check_bf16_encode(orc):
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    xs = u.view(np.float32)
    xs = xs[np.isfinite(xs)]
    # exact ties: a bf16 value plus half its spacing (low 16 bits = 0x8000)
    ties = ((rng.integers(0, 2**16, 4000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    edge = np.array([3.3895314e38, 3.3961776e38, 3.4028235e38, 1e-40, 1e-45, 9.18e-41,
                     1.1754942e-38, 0.0, -0.0, np.inf, -np.inf], dtype=np.float32)
    xs = np.concatenate([xs, ties, edge, -edge])
    ref = bits(torch.from_numpy(xs.copy()).to(torch.bfloat16))
    got = np.array([orc.f32_to_bf16(float(v)) for v in xs], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"f32->bf16 differs for {xs[bad[:5]]}"
    got_nan = orc.f32_to_bf16(float("nan"))
    assert (got_nan & 0x7F80) == 0x7F80 and (got_nan & 0x7F) != 0


# ---------------------------------------------------------------- geometry

def check_output_sizes_golden(orc):
    with open(os.path.join(GOLDEN, "output_sizes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for I, K, S, O in (map(int, r) for r in rows):
        assert orc.fixed_out_size(I, K, S) == O, (I, K, S, O)


def check_fixed_size_by_counting(orc):
    # O is the number of window starts o*S with o*S + K <= I (brute force).
    for I in range(1, 30):
        for K in range(1, 6):
            for S in range(1, 5):
                count = sum(1 for o in range(I + 1) if o * S + K <= I)
                assert orc.fixed_out_size(I, K, S) == count, (I, K, S)


def adaptive_window_exact(i, I, O):
    """floor(i*I/O), ceil((i+1)*I/O) with exact rationals."""
    return math.floor(Fraction(i * I, O)), math.ceil(Fraction((i + 1) * I, O))


def check_adaptive_windows(orc):
    for I in range(1, 41):
        for O in range(1, I + 4):
            prev_start = -1
            covered = set()
            for i in range(O):
                s, e = orc.adaptive_window(i, I, O)
                assert (s, e) == adaptive_window_exact(i, I, O), (i, I, O)
                assert 0 <= s < e <= I and s >= prev_start
                prev_start = s
                covered.update(range(s, e))
                if I % O == 0:
                    assert (s, e) == (i * (I // O), (i + 1) * (I // O))
            assert covered == set(range(I))
            assert orc.adaptive_window(0, I, O)[0] == 0
            assert orc.adaptive_window(O - 1, I, O)[1] == I


def check_fixed_windows(orc):
    for K in range(1, 5):
        for S in range(1, 4):
            for o in range(6):
                assert orc.fixed_window(o, K, S) == (o * S, o * S + K)


# ---------------------------------------------------------------- forward

def _brute_fwd(x: torch.Tensor, wd, wh, ww):
    """Max/argmax per window with numpy's argmax (first occurrence; a NaN
    counts as the maximum) over the row-major ravel of each window box."""
    N, C, D, H, W = x.shape
    xv = x.float().numpy().reshape(N * C, D, H, W)
    xb = bits(x).reshape(N * C, D * H * W)
    out_idx = np.empty((N * C, len(wd), len(wh), len(ww)), dtype=np.int64)
    for p in range(N * C):
        for a, (ds, de) in enumerate(wd):
            for b, (hs, he) in enumerate(wh):
                for c, (ws, we) in enumerate(ww):
                    box = xv[p, ds:de, hs:he, ws:we]
                    k = int(np.argmax(box.ravel()))
                    dd, hh, wq = np.unravel_index(k, box.shape)
                    out_idx[p, a, b, c] = ((ds + dd) * H + hs + hh) * W + ws + wq
    ybits = np.take_along_axis(xb, out_idx.reshape(N * C, -1), axis=1)
    return ybits.reshape(-1), out_idx.reshape(-1)


def _tie_heavy(rng, shape, dtype):
    """Small integers (many ties), with some -0/+0 and a few NaNs."""
    x = torch.from_numpy(rng.integers(-3, 4, size=shape).astype(np.float32))
    flat = x.view(-1)
    n = flat.numel()
    zeros = torch.from_numpy(rng.choice(n, size=max(1, n // 8), replace=False))
    flat[zeros] = torch.where(torch.from_numpy(rng.random(zeros.numel()) < 0.5),
                              torch.tensor(-0.0), torch.tensor(0.0))
    if rng.random() < 0.5:
        nans = torch.from_numpy(rng.choice(n, size=max(1, n // 40), replace=False))
        flat[nans] = float("nan")
    return x.to(dtype)


def _random_input(rng, shape, dtype):
    if rng.random() < 0.6:
        return _tie_heavy(rng, shape, dtype)
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(dtype)


def check_fwd_bruteforce_fixed(orc, cases=80, seed=1):
    rng = np.random.default_rng(seed)
    for t in range(cases):
        D, H, W = (int(v) for v in rng.integers(1, 7, 3))
        K = [int(rng.integers(1, min(I, 4) + 1)) for I in (D, H, W)]
        S = [int(v) for v in rng.integers(1, 4, 3)]
        N, C = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        dtype = DTYPES[t % 3]
        x = _random_input(rng, (N, C, D, H, W), dtype)
        wins = []
        for I, k, s in zip((D, H, W), K, S):
            wins.append([(o * s, o * s + k) for o in range(I) if o * s + k <= I])
        y, idx = orc.maxpool3d_fwd(x, K, S)
        assert tuple(y.shape[2:]) == tuple(len(w) for w in wins)
        yb, ib = _brute_fwd(x, *wins)
        assert np.array_equal(idx.numpy().reshape(-1), ib), (D, H, W, K, S, dtype)
        assert np.array_equal(bits(y).reshape(-1), yb)


def check_fwd_bruteforce_adaptive(orc, cases=80, seed=2):
    rng = np.random.default_rng(seed)
    for t in range(cases):
        D, H, W = (int(v) for v in rng.integers(1, 7, 3))
        O = [int(rng.integers(1, I + 3)) for I in (D, H, W)]
        N, C = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        dtype = DTYPES[t % 3]
        x = _random_input(rng, (N, C, D, H, W), dtype)
        wins = [[adaptive_window_exact(i, I, o) for i in range(o)] for I, o in zip((D, H, W), O)]
        y, idx = orc.adaptive_maxpool3d_fwd(x, O)
        yb, ib = _brute_fwd(x, *wins)
        assert np.array_equal(idx.numpy().reshape(-1), ib), (D, H, W, O, dtype)
        assert np.array_equal(bits(y).reshape(-1), yb)


def check_fwd_hand_examples(orc):
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        g = json.load(f)
    x = torch.tensor(g["x"], dtype=torch.float32).reshape(1, 1, 2, 2, 4)
    for case in g["cases"]:
        for dtype in DTYPES:
            y, idx = orc.maxpool3d_fwd(x.to(dtype), case["kernel"], case["stride"])
            assert y.float().reshape(-1).tolist() == case["y"], case["name"]
            assert idx.reshape(-1).tolist() == case["idx"], case["name"]


def check_fwd_identity(orc):
    rng = np.random.default_rng(3)
    for dtype in DTYPES:
        x = _random_input(rng, (2, 3, 3, 4, 5), dtype)
        ref_idx = np.tile(np.arange(60), 6)
        for y, idx in (orc.adaptive_maxpool3d_fwd(x, (3, 4, 5)),
                       orc.maxpool3d_fwd(x, (1, 1, 1), (1, 1, 1))):
            assert np.array_equal(bits(y).reshape(-1), bits(x).reshape(-1))
            assert np.array_equal(idx.numpy().reshape(-1), ref_idx)


def check_fixed_equals_divisible_adaptive(orc):
    rng = np.random.default_rng(4)
    for t in range(24):
        K = [int(v) for v in rng.integers(1, 4, 3)]
        O = [int(v) for v in rng.integers(1, 4, 3)]
        I = [k * o for k, o in zip(K, O)]
        x = _random_input(rng, (1, 2) + tuple(I), DTYPES[t % 3])
        y1, i1 = orc.maxpool3d_fwd(x, K, K)
        y2, i2 = orc.adaptive_maxpool3d_fwd(x, O)
        assert np.array_equal(bits(y1), bits(y2)) and torch.equal(i1, i2)


# ---------------------------------------------------------------- backward

def _random_idx_in_windows(rng, P, wins, H, W):
    """An index per window, drawn uniformly from the window's cells."""
    wd, wh, ww = wins
    idx = np.empty((P, len(wd), len(wh), len(ww)), dtype=np.int64)
    for p, a, b, c in itertools.product(range(P), range(len(wd)), range(len(wh)), range(len(ww))):
        d = int(rng.integers(*wd[a]))
        h = int(rng.integers(*wh[b]))
        w = int(rng.integers(*ww[c]))
        idx[p, a, b, c] = (d * H + h) * W + w
    return idx


def check_bwd_hand_examples(orc):
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        n = len(case["idx"])
        idx = torch.tensor(case["idx"], dtype=torch.int64).reshape(1, 1, 1, 1, n)
        for dtype in DTYPES:
            go = torch.tensor(case["grad_out"], dtype=dtype).reshape(1, 1, 1, 1, n)
            gin = orc.maxpool3d_bwd(go, idx, (2, 2, 4))
            assert gin.float().reshape(-1).tolist() == case["grad_in"], case["name"]
    for case in g["order_cases"]:
        dtype = getattr(torch, case["dtype"])
        go = torch.tensor(case["grad_out"], dtype=dtype).reshape(1, 1, 1, 1, 3)
        idx = torch.full((1, 1, 1, 1, 3), 2, dtype=torch.int64)
        gin = orc.maxpool3d_bwd(go, idx, (1, 1, 5))
        assert gin.float().reshape(-1).tolist() == [0, 0, case["grad_in_at_2"], 0, 0], case["name"]


def check_bwd_disjoint_bijection(orc):
    """Disjoint windows: every window's gradient lands once, bit for bit, at
    its index; every other input holds +0."""
    rng = np.random.default_rng(5)
    for t in range(30):
        K = [int(v) for v in rng.integers(1, 4, 3)]
        S = [k + int(rng.integers(0, 2)) for k in K]           # kernel <= stride
        D, H, W = (k + int(rng.integers(0, 6)) for k in K)
        wins = [[(o * s, o * s + k) for o in range(I) if o * s + k <= I]
                for I, k, s in zip((D, H, W), K, S)]
        P = 3
        idx = _random_idx_in_windows(rng, P, wins, H, W)
        dtype = DTYPES[t % 3]
        nout = idx[0].size
        go = torch.arange(1, P * nout + 1, dtype=torch.float32).reshape(idx.shape) * 0.25
        go = go.to(dtype).reshape((1, P) + idx.shape[1:])
        gin = orc.maxpool3d_bwd(go, torch.from_numpy(idx).reshape(go.shape), (D, H, W))
        gb = bits(gin).reshape(P, -1)
        ob = bits(go).reshape(P, -1)
        expect = np.zeros_like(gb)
        for p in range(P):
            expect[p, idx[p].reshape(-1)] = ob[p]
        assert np.array_equal(gb, expect)


def _overlap_case(rng, t):
    K = [int(v) for v in rng.integers(2, 5, 3)]
    S = [max(1, k - int(rng.integers(1, 3))) for k in K]      # stride < kernel
    D, H, W = (k + int(rng.integers(0, 6)) for k in K)
    wins = [[(o * s, o * s + k) for o in range(I) if o * s + k <= I]
            for I, k, s in zip((D, H, W), K, S)]
    return (D, H, W), wins


def check_bwd_integer_sum_conserved(orc):
    """Integer-valued gradients: every partial sum is exact, so the total of
    grad_in equals the total of grad_out, per plane."""
    rng = np.random.default_rng(6)
    for t in range(30):
        (D, H, W), wins = _overlap_case(rng, t)
        P = 2
        idx = _random_idx_in_windows(rng, P, wins, H, W)
        go = torch.from_numpy(rng.integers(-20, 21, size=idx.shape).astype(np.float32))
        go = go.to(DTYPES[t % 3]).reshape((1, P) + idx.shape[1:])
        gin = orc.maxpool3d_bwd(go, torch.from_numpy(idx).reshape(go.shape), (D, H, W))
        s_in = gin.double().reshape(P, -1).sum(1)
        s_out = go.double().reshape(P, -1).sum(1)
        assert torch.equal(s_in, s_out)


def check_bwd_against_exact_sum(orc):
    """Against math.fsum of each input's contributions: within the error
    bound of a left-to-right binary32 sum plus one final rounding; a single
    contribution is copied exactly; inputs nobody selects are +0."""
    rng = np.random.default_rng(8)
    half_ulp = {torch.float32: 2.0**-24, torch.float16: 2.0**-11, torch.bfloat16: 2.0**-8}
    tiny = {torch.float32: 2.0**-150, torch.float16: 2.0**-25, torch.bfloat16: 2.0**-134}
    for t in range(30):
        (D, H, W), wins = _overlap_case(rng, t)
        P = 2
        dtype = DTYPES[t % 3]
        idx = _random_idx_in_windows(rng, P, wins, H, W)
        go = torch.from_numpy(rng.standard_normal(idx.shape).astype(np.float32)).to(dtype)
        go = go.reshape((1, P) + idx.shape[1:])
        gin = orc.maxpool3d_bwd(go, torch.from_numpy(idx).reshape(go.shape), (D, H, W))
        gv = go.double().reshape(P, -1).numpy()
        gi = gin.double().reshape(P, -1).numpy()
        gib = bits(gin).reshape(P, -1)
        gob = bits(go).reshape(P, -1)
        for p in range(P):
            terms = {}
            for o, j in enumerate(idx[p].reshape(-1)):
                terms.setdefault(int(j), []).append(o)
            for j in range(D * H * W):
                os_ = terms.get(j, [])
                if not os_:
                    assert gib[p, j] == 0            # +0 exactly
                elif len(os_) == 1:
                    assert gib[p, j] == gob[p, os_[0]]
                else:
                    vals = [gv[p, o] for o in os_]
                    exact = math.fsum(vals)
                    sabs = math.fsum(abs(v) for v in vals)
                    tol = (len(vals) - 1) * 2.0**-24 * sabs
                    tol += half_ulp[dtype] * (abs(exact) + tol) + tiny[dtype]
                    assert abs(gi[p, j] - exact) <= tol, (p, j, gi[p, j], exact, tol)


def check_bwd_signed_zero(orc):
    """Sums of signed zeros, with the sign IEEE 754 (section 6.3) fixes for
    a sum in round-to-nearest: a lone contribution is the gradient itself
    (the disjoint gather writes it bit for bit, [AMPB] Summary), so a lone
    -0 stays -0; -0 + -0 is -0; zeros of opposite signs, in either order,
    and an exact cancellation x + (-x) give +0; an input nobody selects is
    +0. Expected values are written out per case, not computed."""
    NEG, POS = -0.0, 0.0
    # (contributions in ascending output order, expected result)
    cases = [
        ([NEG], NEG),
        ([NEG, NEG], NEG),
        ([NEG, POS], POS),
        ([POS, NEG], POS),
        ([NEG, NEG, NEG], NEG),
        ([1.5, -1.5], POS),
        ([-1.5, 1.5, NEG], POS),
        ([NEG, 2.0, -2.0], POS),
        ([], POS),
    ]
    targets, grads = [], []
    # interleave the inputs' contributions so that each input's terms are
    # spread over the output order
    longest = max(len(c) for c, _ in cases)
    for k in range(longest):
        for j, (terms, _) in enumerate(cases):
            if k < len(terms):
                targets.append(j)
                grads.append(terms[k])
    n = len(grads)
    idx = torch.tensor(targets, dtype=torch.int64).reshape(1, 1, 1, 1, n)
    for dtype in DTYPES:
        go = torch.tensor(grads, dtype=torch.float32).to(dtype).reshape(1, 1, 1, 1, n)
        gin = orc.maxpool3d_bwd(go, idx, (1, 1, len(cases)))
        got = gin.float().reshape(-1).tolist()
        for j, (terms, want) in enumerate(cases):
            assert got[j] == want and math.copysign(1.0, got[j]) == math.copysign(1.0, want), (
                dtype, terms, got[j], want)


# ----------------------------------------------------- padding and dilation
# The forward with padding, dilation and ceil mode against torch's CPU
# max_pool1d / max_pool3d (a library routine whose tie rule, for values
# that are not NaN, is the same: a later element replaces only when it is
# strictly greater).

def _torch_len(I, K, S, p, dl, ceil_mode):
    """torch's output length, or 0 when torch rejects the arguments."""
    try:
        return torch.nn.functional.max_pool1d(torch.zeros(1, 1, I), K, S, p, dl, ceil_mode).shape[-1]
    except RuntimeError:
        return 0


def check_ex_out_size_vs_torch(orc):
    for I, K, S, p, dl, cm in itertools.product(range(1, 11), range(1, 5), range(1, 4), range(0, 3),
                                                 range(1, 4), (False, True)):
        got = orc.ex_out_size(I, K, S, p, dl, cm)
        want = _torch_len(I, K, S, p, dl, cm)
        assert got == max(want, 0), (I, K, S, p, dl, cm, got, want)


def _ex_cases(rng, n):
    out = []
    while len(out) < n:
        k = [int(v) for v in rng.integers(1, 4, 3)]
        s = [int(v) for v in rng.integers(1, 4, 3)]
        dl = [int(v) for v in rng.integers(1, 3, 3)]
        p = [int(rng.integers(0, kk // 2 + 1)) for kk in k]
        shape = (1, 2) + tuple(int(v) for v in rng.integers(1, 9, 3))
        cm = bool(rng.integers(0, 2))
        out.append((shape, tuple(k), tuple(s), tuple(p), tuple(dl), cm))
    return out


def check_fwd_ex_vs_torch(orc, cases=120, seed=11):
    rng = np.random.default_rng(seed)
    checked = 0
    for shape, k, s, p, dl, cm in _ex_cases(rng, cases):
        n = int(np.prod(shape))
        for kind in ("distinct", "ties"):
            if kind == "distinct":
                x = torch.from_numpy(rng.permutation(n).astype(np.float32)).reshape(shape) / n - 0.5
            else:
                x = torch.from_numpy(rng.integers(-2, 3, n).astype(np.float32)).reshape(shape)
            try:
                yt, it = torch.nn.functional.max_pool3d(x, k, s, p, dl, cm, True)
            except RuntimeError:
                assert min(orc.ex_out_size(I, kk, ss, pp, dd, cm)
                           for I, kk, ss, pp, dd in zip(shape[2:], k, s, p, dl)) == 0
                continue
            try:
                y, i = orc.maxpool3d_fwd_ex(x, k, s, p, dl, cm)
            except (RuntimeError, ValueError):
                # a window with no position inside the input: torch leaves -inf there
                assert bool(torch.isinf(yt).any()), (shape, k, s, p, dl, cm)
                continue
            assert torch.equal(i, it), (shape, k, s, p, dl, cm, kind)
            assert np.array_equal(bits(y), bits(yt)), (shape, k, s, p, dl, cm, kind)
            checked += 1
    assert checked >= cases


def check_fwd_ex_16bit_vs_torch(orc, cases=40, seed=12):
    rng = np.random.default_rng(seed)
    for shape, k, s, p, dl, cm in _ex_cases(rng, cases):
        for dtype in (torch.float16, torch.bfloat16):
            n = int(np.prod(shape))
            x = torch.from_numpy(rng.integers(-3, 4, n).astype(np.float32)).reshape(shape).to(dtype)
            try:
                yt, it = torch.nn.functional.max_pool3d(x, k, s, p, dl, cm, True)
                y, i = orc.maxpool3d_fwd_ex(x, k, s, p, dl, cm)
            except (RuntimeError, ValueError):
                continue
            assert torch.equal(i, it), (shape, k, s, p, dl, cm, dtype)
            assert np.array_equal(bits(y), bits(yt)), (shape, k, s, p, dl, cm, dtype)


def check_fwd_ex_reduces_to_plain(orc, seed=13):
    rng = np.random.default_rng(seed)
    for _ in range(30):
        k = tuple(int(v) for v in rng.integers(1, 4, 3))
        s = tuple(int(v) for v in rng.integers(1, 4, 3))
        shape = (2, 2) + tuple(int(kk + rng.integers(0, 6)) for kk in k)
        x = torch.from_numpy(rng.standard_normal(int(np.prod(shape))).astype(np.float32)).reshape(shape)
        y0, i0 = orc.maxpool3d_fwd(x, k, s)
        y1, i1 = orc.maxpool3d_fwd_ex(x, k, s, (0, 0, 0), (1, 1, 1), False)
        assert torch.equal(i0, i1) and np.array_equal(bits(y0), bits(y1))


ALL_CHECKS = [
    check_f16_decode, check_f16_encode, check_bf16_decode, check_bf16_encode,
    check_output_sizes_golden, check_fixed_size_by_counting, check_adaptive_windows,
    check_fixed_windows, check_fwd_bruteforce_fixed, check_fwd_bruteforce_adaptive,
    check_fwd_hand_examples, check_fwd_identity, check_fixed_equals_divisible_adaptive,
    check_bwd_hand_examples, check_bwd_disjoint_bijection, check_bwd_integer_sum_conserved,
    check_bwd_against_exact_sum, check_bwd_signed_zero, check_ex_out_size_vs_torch, check_fwd_ex_vs_torch,
    check_fwd_ex_16bit_vs_torch, check_fwd_ex_reduces_to_plain,
]
