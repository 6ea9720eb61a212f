"""Host logic of bench.py that needs no GPU: the traffic record applies only
to the whole workload it was taken on and only on the sources it was taken
on, and both arms print the same config object."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bwd_maxpool3d_fwd_gb300 import workloads  # noqa: E402


def test_traffic_record_scope(monkeypatch):
    # each kernel's record applies only to the whole workload it was taken on
    # and only while that kernel's sources are the ones it was taken on
    name = bench.TRAFFIC_WORKLOAD
    for kind in ("fwd", "bwd"):
        full = bench.recorded_traffic(kind, name, True)
        if full is None:      # taken on other sources of this kernel: nothing applies
            continue
        assert full > 0
        assert bench.recorded_traffic(kind, name, False) is None         # a subset of planes
        assert bench.recorded_traffic(kind, "adaptive_f16_16x64x30x50x50_to_8x12x12", True) is None
        with monkeypatch.context() as m:
            m.setattr(bench, "kernel_hash", lambda k: "000000000000")
            assert bench.recorded_traffic(kind, name, True) is None      # other sources


def test_workload_config_keys():
    w = workloads.WORKLOADS[bench.HEADLINE]
    cfg = bench.workload_config(w, "ncdhw", 1)
    assert cfg["workload"] == w.name == bench.TRAFFIC_WORKLOAD
    assert set(cfg) == {"workload", "input", "output", "kernel", "stride", "padding", "layout", "l2",
                        "parallelism"}
    assert cfg["input"] == [32, 128, 16, 112, 112] and cfg["output"] == [32, 128, 7, 55, 55]
