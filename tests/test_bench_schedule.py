"""bench.py's schedule record (CPU): the ring utilisation of each benchmark
workload's partition, taken from dfa_make_schedule.  A P-worker causal
ring over contiguous chunks keeps (P + 1) / 2 of P^2 slots busy and, in
lockstep, pays the diagonal's half pair on every step; the folded and
striped partitions give every worker the same load on every step (Striped
Attention Guide, "Workload Balance Theorem"; DistFlashAttn Guide, "The
Causal Imbalance Crisis")."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from long_context_flashattention_gb300.inputs import WORKLOADS  # noqa: E402


def test_contiguous_ring_closed_forms():
    N, P = 131072, 8
    s = bench.schedule_summary(N, P, "contiguous")
    assert s["total_pairs"] == N * (N + 1) // 2
    assert s["eta_slots"] == pytest.approx((P + 1) / (2 * P))
    # lockstep: every step's busiest worker holds a full chunk pair (C^2), the
    # first step a diagonal one (C (C + 1) / 2)
    C = N // P
    busiest = C * (C + 1) // 2 + (P - 1) * C * C
    assert s["eta_flops"] == pytest.approx(s["total_pairs"] / (P * busiest), abs=1e-6)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_benchmark_partitions_are_balanced(name):
    w = WORKLOADS[name]
    kind = w.partitions[0]
    s = bench.schedule_summary(w.N, w.P, kind)
    assert s["total_pairs"] == w.N * (w.N + 1) // 2
    if kind in ("balanced", "striped"):
        assert s["eta_slots"] == 1.0
        assert s["eta_flops"] > 0.999
