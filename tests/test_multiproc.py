"""Host logic of the multi-GPU benchmark path with two gloo ranks on CPU:
the process group comes up from the torchrun-style environment, the max
over ranks picks the slowest rank's time, and each rank's shard is an
independent instance of the workload (different seed, same shapes)."""
import os
import socket

import pytest
import torch.multiprocessing as tmp

pytestmark = pytest.mark.timeout(120) if hasattr(pytest.mark, "timeout") else []


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    from bwd_maxpool3d_fwd_gb300 import workloads
    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    mx = bench.max_over_ranks(10.0 + rank, w, "cpu")
    shard = bench.shard_seed(workloads.WORKLOADS[0], rank)
    x = workloads.make_x(shard)
    out[rank] = (mx, shard.seed, tuple(x.reshape(-1)[:8].tolist()), tuple(x.shape))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = tmp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (m0, s0, x0, sh0), (m1, s1, x1, sh1) = out[0], out[1]
    assert m0 == m1 == 11.0                 # the slowest rank's time
    assert s0 != s1 and x0 != x1            # independent shards
    assert sh0 == sh1                       # of the same workload shape
