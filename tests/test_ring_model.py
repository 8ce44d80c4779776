"""The flat / hierarchical ring step model against the pages' printed
forward-latency breakdown (tests/golden/ring_latency_mtraining.txt)."""
import os

import pytest

from dynamic_sparse_attention_index_gb300 import ring_model as rm

GOLD = os.path.join(os.path.dirname(__file__), "golden", "ring_latency_mtraining.txt")


def _gold():
    out = {}
    for ln in open(GOLD):
        ln = ln.strip()
        if ln and not ln.startswith("#"):
            k, v = ln.split()
            out[k] = float(v)
    return out


def test_pages_breakdown_reproduced():
    g = _gold()
    topo = rm.RingTopology(int(g["nodes"]), int(g["gpus_per_node"]), g["t_intra"], g["t_inter"])
    comp = [g["t_comp"]] * topo.workers
    r = rm.forward_latency_ms(comp, topo, index_ms=g["index_build"], other_ms=g["cpu_ops"])
    f, h = r["flat"], r["hierarchical"]
    assert sum(f["steps_ms"][:-1]) == pytest.approx(g["flat_ring_steps"], abs=1e-9)
    assert f["steps_ms"][-1] == pytest.approx(g["flat_last_compute"])
    assert r["flat_ms"] == pytest.approx(g["flat_total"], abs=1e-9)
    assert h["total_ms"] == pytest.approx(g["hier_ring_steps"], abs=1e-9)
    assert r["hierarchical_ms"] == pytest.approx(g["hier_total"], abs=1e-9)
    assert 100 * r["reduction"] == pytest.approx(g["reduction_percent"], abs=0.05)
    assert f["comm_bound_steps"] == 31 and h["exposed_outer_ms"] == 0.0


def test_limits():
    topo = rm.RingTopology(4, 8, 0.13, 0.98)
    # compute slower than every link: both schedules are the sum of compute
    comp = [2.0 + 0.01 * t for t in range(32)]
    assert rm.flat_ring_ms(comp, topo)["total_ms"] == pytest.approx(sum(comp))
    assert rm.hierarchical_ring_ms(comp, topo)["total_ms"] == pytest.approx(sum(comp))
    # one node: the flat ring is NVLink bound only
    one = rm.RingTopology(1, 8, 0.13, 0.98)
    comp = [0.05] * 8
    assert rm.flat_ring_ms(comp, one)["total_ms"] == pytest.approx(7 * 0.13 + 0.05)
    # tiny compute: each hierarchical round waits for the outer transfer
    fast = rm.RingTopology(4, 8, 0.05, 0.98)
    comp = [0.01] * 32
    h = rm.hierarchical_ring_ms(comp, fast)
    assert h["total_ms"] == pytest.approx(3 * 0.98 + 8 * 0.05)
    assert h["exposed_outer_ms"] == pytest.approx(3 * (0.98 - 8 * 0.05))


def test_step_compute_is_slowest_worker():
    t = [[1.0, 2.0, 0.5], [3.0, 1.0, 0.5], [2.0, 2.5, 4.0]]
    assert rm.step_compute_ms(t) == [3.0, 2.5, 4.0]
