"""The give-up path of the forward kernels' bounded copy waits (needs a GPU).

The stride-2 forward and the plane-pair depth walk stream input slices into
shared memory with bulk copies and wait for each on an mbarrier, giving up
after a bounded number of polls. Lowering that bound to 0 through
mp3d_set_pipeline_wait_limit makes every such wait give up at once, without
any fault or unbounded wait: the kernels still let their copies in flight
land (those waits keep the normal bound) before they exit. Each case checks
that the call returns, that bit 0 of the device error flags is raised and
can be cleared, and that the next call with the normal bound matches the
oracle bit for bit. A bound of 1 poll lets some waits succeed, so the walk
gives up part way through.
"""
import ctypes

import pytest
import torch

import bwd_maxpool3d_fwd_gb300 as mp
import oracle
from gpu_helpers import DEV, assert_bits_equal

pytestmark = pytest.mark.gpu

CASES = [
    # (name, input shape, forward kind, window args, expected path)
    ("stride2_k3s2", (2, 3, 9, 30, 64), "fixed", ((3, 3, 3), (2, 2, 2)), "fwd_s2"),
    ("pair_adaptive", (2, 4, 30, 50, 50), "adaptive", (8, 12, 12), "fwd_roll"),
    ("pair_padded", (2, 4, 16, 50, 50), "padded", ((3, 3, 3), (2, 2, 2), (1, 1, 1)), "fwd_roll"),
    ("stride2_padded", (2, 4, 16, 56, 56), "padded", ((3, 3, 3), (2, 2, 2), (1, 1, 1)), "fwd_s2"),
]


def set_limit(polls: int) -> int:
    f = mp.lib().mp3d_set_pipeline_wait_limit
    f.argtypes = [ctypes.c_int]
    f.restype = ctypes.c_int
    return f(polls)


def forward(kind, x, args):
    if kind == "fixed":
        k, s = args
        out = mp.pool_out_size(x.shape[2:], k, s)
    elif kind == "adaptive":
        out = tuple(args)
    else:
        k, s, p = args
        out = mp.pool_out_size_ex(x.shape[2:], k, s, p)
    y = torch.empty(x.shape[:2] + out, dtype=x.dtype, device=DEV)
    idx = torch.empty(x.shape[:2] + out, dtype=torch.int64, device=DEV)
    if kind == "fixed":
        mp.maxpool3d_fwd(x, y, idx, *args)
    elif kind == "adaptive":
        mp.adaptive_maxpool3d_fwd(x, y, idx, args)
    else:
        mp.maxpool3d_fwd_ex(x, y, idx, *args)
    torch.cuda.synchronize()
    return y, idx


def plan(kind, shape, args, dtype):
    if kind == "fixed":
        return mp.maxpool3d_fwd_plan(shape, *args, dtype)
    if kind == "adaptive":
        return mp.adaptive_maxpool3d_fwd_plan(shape, args, dtype)
    k, s, p = args
    return mp.maxpool3d_fwd_ex_plan(shape, k, s, p, (1, 1, 1), False, dtype)


def reference(kind, x, args):
    if kind == "fixed":
        return oracle.maxpool3d_fwd(x, *args)
    if kind == "adaptive":
        return oracle.adaptive_maxpool3d_fwd(x, args)
    k, s, p = args
    return oracle.maxpool3d_fwd_ex(x, k, s, p, (1, 1, 1), False)


@pytest.mark.parametrize("polls", [0, 1])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_wait_give_up_then_recover(case, polls):
    name, shape, kind, args, path = case
    dtype = torch.float16
    assert plan(kind, shape, args, dtype) == path
    gen = torch.Generator().manual_seed(71)
    x = torch.randn(shape, generator=gen).to(dtype)
    y_ref, i_ref = reference(kind, x, args)
    xd = x.to(DEV)
    assert mp.mp3d_device_error_flags(clear=True) == 0
    prev = set_limit(polls)
    try:
        forward(kind, xd, args)          # returns; its outputs are not used
    finally:
        set_limit(prev)
    flags = mp.mp3d_device_error_flags(clear=True)
    if polls == 0:
        assert flags & 1, "every wait gave up, so the flag must be raised"
    assert mp.mp3d_device_error_flags(clear=False) == 0, "flags cleared"
    # the normal bound again: exact results, no flag
    y, idx = forward(kind, xd, args)
    assert torch.equal(idx.cpu(), i_ref)
    assert_bits_equal(y.cpu(), y_ref, f"y after the give-up path ({name})")
    assert mp.mp3d_device_error_flags(clear=False) == 0

