"""bench.py reports DRAM traffic only from a committed ncu summary that matches (CPU)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from split_bf16_gemm_swap_gb300 import lowm  # noqa: E402

WORKLOADS = [bench.WORKLOAD, bench.WIDE] + [dict(M=M, N=N, K=K, split_k=sk) for _, (M, N, K, sk) in
                                             bench.OTHER_CONFIGS]


def tactic(w):
    # the benchmark times every workload with the W-before-PDL promise
    st, t = lowm.lowm_gemm_query_tactic_ex(w["M"], w["N"], w["K"], w["split_k"], lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    assert st == lowm.LOWM_OK
    return t


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: "M%d_N%d_K%d" % (w["M"], w["N"], w["K"]))
def test_committed_profiles_match_the_current_device_code(w):
    # Every workload bench.py times has a committed ncu summary of the current
    # device code and tactic, so its line carries the measured DRAM traffic.
    t = tactic(w)
    got = bench.committed_traffic(dict(w, split_k=t["split_k"]), t)
    assert got is not None
    algo = bench.algo_bytes(w["M"], w["N"], w["K"])
    assert 0.95 * algo <= got <= 1.02 * algo          # no re-reads (A and C may stay in L2)


def test_traffic_is_withheld_when_the_ring_differs():
    t = dict(tactic(bench.WORKLOAD))
    t["stages"] += 1
    assert bench.committed_traffic(bench.WORKLOAD, t) is None


def test_traffic_is_withheld_when_the_tile_width_differs():
    t = dict(tactic(bench.WORKLOAD))
    t["tile_n"] = 64 if t["tile_n"] == 128 else 128
    assert bench.committed_traffic(bench.WORKLOAD, t) is None


def test_traffic_is_withheld_when_the_device_code_changed(monkeypatch):
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "0000000000000000")
    assert bench.committed_traffic(bench.WORKLOAD, tactic(bench.WORKLOAD)) is None


def test_traffic_is_withheld_for_a_workload_without_a_summary():
    assert bench.committed_traffic(dict(M=3, N=640, K=1024, split_k=2),
                                   {"kb_per_stage": 4, "stages": 2, "tile_n": 64}) is None
