"""The byte accounting bench.py divides by: the compulsory bytes of one
forward (w, sh, src per edge; one read of x, one write of out and the row
pointers per node) and of one fp32 backward, checked against the totals the
scope table states for each workload (0.919 / 6.72 / 8.29 GB forward, 1.82 GB
backward) on the seeded graphs the benchmark builds."""
import os
import sys
from types import SimpleNamespace

import pytest

from oracle import tp
from workloads import WORKLOADS, make_graph

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _desc(wl):
    pl = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    return SimpleNamespace(weight_numel=pl.weight_numel, dim_sh=pl.dim_sh, dim_x=pl.dim_in, dim_out=pl.dim_out)


@pytest.mark.parametrize("name,total_gb", [("medium", 0.919), ("large", 6.72), ("xlarge", 8.29)])
def test_forward_compulsory_bytes(name, total_gb):
    import bench
    wl = WORKLOADS[name]
    _, src, _, _, n = make_graph(wl, 0)
    esz = 2 if wl.dtype == "bf16" else 4
    got = bench.algorithmic_bytes(_desc(wl), n, len(src), esz) / 1e9
    assert got == pytest.approx(total_gb, rel=0.01)


def test_backward_compulsory_bytes():
    import bench
    wl = WORKLOADS["medium"]
    _, src, _, _, n = make_graph(wl, 0)
    assert bench.backward_bytes(_desc(wl), n, len(src)) / 1e9 == pytest.approx(1.82, rel=0.01)
