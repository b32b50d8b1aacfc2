"""bench.py reports DRAM traffic only from a committed ncu summary that matches (CPU)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_committed_profiles_match_the_current_device_code():
    # Every committed kernel summary was taken on the current device code, so
    # the headline and wide-N lines carry their traffic.
    head = bench.committed_traffic(bench.WORKLOAD, {"kb_per_stage": 4, "stages": 3})
    wide = bench.committed_traffic(bench.WIDE, {"kb_per_stage": 2, "stages": 2})
    for got, w in ((head, bench.WORKLOAD), (wide, bench.WIDE)):
        assert got is not None
        algo = bench.algo_bytes(w["M"], w["N"], w["K"])
        assert algo <= got <= 1.02 * algo          # ncu saw no re-reads


def test_traffic_is_withheld_when_the_ring_differs():
    assert bench.committed_traffic(bench.WORKLOAD, {"kb_per_stage": 2, "stages": 3}) is None


def test_traffic_is_withheld_when_the_device_code_changed(monkeypatch):
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "0000000000000000")
    assert bench.committed_traffic(bench.WORKLOAD, {"kb_per_stage": 4, "stages": 3}) is None


def test_traffic_is_withheld_for_a_workload_without_a_summary():
    assert bench.committed_traffic(dict(M=3, N=640, K=1024, split_k=2), {"kb_per_stage": 4, "stages": 2}) is None
