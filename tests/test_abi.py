"""The C-ABI library builds, loads and exports what include/lowm_gemm.h declares.

CPU-only: no call here touches a GPU.  Host-side argument checks that run
before any device query (null and misaligned pointers, bad sizes) and the
host-only tactic query are exercised directly.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from split_bf16_gemm_swap_gb300 import build, lowm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lowm_gemm.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return lowm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(lowm_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_binding_functions():
    assert tuple(declared_functions()) == lowm.ABI_FUNCTIONS


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings(L):
    for s in range(7):
        assert lowm.status_string(s)
    assert "unknown" in lowm.status_string(99)


def test_shipped_tactic_is_reproduced(L, monkeypatch):
    # The pages' tactic (64, 8, 2, 10): 64-column tiles, m_pad 8, split_k 2, 10
    # single-block stages.
    monkeypatch.setenv("LOWM_TILE_N", "64")
    monkeypatch.setenv("LOWM_KB_PER_STAGE", "1")
    monkeypatch.setenv("LOWM_STAGES", "10")
    st, t = lowm.lowm_gemm_query_tactic(4, 6144, 4096, 2)
    assert st == lowm.LOWM_OK
    assert (t["tile_n"], t["m_pad"], t["split_k"], t["stages"], t["block_k"]) == (64, 8, 2, 10, 64)
    assert t["num_clusters"] == 96 and t["ctas"] == 192 and t["pdl"] == 1 and t["persistent"] == 0


def test_default_tactic_for_the_headline_workload(L):
    # GB300: 128-column tiles, one CTA per SM on 96 SMs, a 4 x 3 ring (192 KiB
    # of W) that fits only with the mailbox in the ring, the whole ring
    # requested before the dependency wait: 8.90 us, against 9.53 us for the
    # 4 x 2 ring and 10.14 us for 64-column tiles on 192 CTAs.
    st, t = lowm.lowm_gemm_query_tactic_ex(4, 6144, 4096, 2, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    assert st == lowm.LOWM_OK
    assert (t["tile_n"], t["m_pad"], t["split_k"], t["kb_per_stage"], t["stages"]) == (128, 16, 2, 4, 3)
    assert t["num_clusters"] == 48 and t["ctas"] == 96 and t["persistent"] == 0 and t["smem_bytes"] <= 232448
    assert t["l2_prefetch_stages"] == 1 and t["mbox_in_ring"] == 1 and t["w_prefetch_stages"] == 3
    # Without the W promise (lowm_gemm_bf16) the deeper ring measured slower: the 4 x 2 ring next to the
    # mailbox, 10.67 us against 11.17 us.
    st, t0 = lowm.lowm_gemm_query_tactic(4, 6144, 4096, 2)
    assert st == lowm.LOWM_OK and (t0["tile_n"], t0["kb_per_stage"], t0["stages"], t0["mbox_in_ring"]) == (128, 4, 2, 0)


@pytest.mark.parametrize("M,N,K,sk,tile", [
    # GB300, W promise, 64 -> 128 columns (us): 128 columns on 64 to two-per-SM CTAs with short streams
    (4, 6144, 4096, 2, 128), (16, 6144, 4096, 2, 128), (32, 6144, 4096, 2, 128), (64, 6144, 4096, 2, 128),
    (128, 6144, 4096, 2, 128),    # 10.14 -> 9.43 at M4
    (4, 2304, 12288, 4, 128),     # 72 CTAs of 768 KiB: 9.97 -> 9.67
    (4, 4096, 4096, 2, 128),      # 64 CTAs: 7.36 -> 6.79
    (4, 6144, 4096, 4, 128),      # 192 CTAs, two per SM: 9.72 -> 9.21
    (16, 6144, 32768, 4, 128),    # 192 CTAs of 2 MiB, a CTA on every SM: 62.5 -> 61.1
    (4, 2304, 12288, 2, 64),      # 36 CTAs: 11.96 -> 15.77
    (4, 2304, 12288, 8, 64),      # split_k 8: 13.1 -> 15.0
    (4, 49152, 4096, 2, 64),      # four CTAs per SM: 61.1 -> 67.1
    (4, 8192, 8192, 1, 64),       # 64 CTAs of 2 MiB: 21.6 -> 25.3
    (16, 6144, 32768, 2, 64),     # 96 CTAs of 4 MiB
    (64, 6144, 4096, 4, 64),      # m_pad 64, split_k 4, two per SM: 17.4 -> 21.1
    (64, 2304, 12288, 4, 64),     # m_pad 64 where the 64-column grid fits: 12.47 -> 13.84
    (4, 6152, 4096, 2, 64)])      # N not a multiple of 128
def test_tile_width_rule(L, M, N, K, sk, tile):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    assert st == lowm.LOWM_OK and t["tile_n"] == tile


@pytest.mark.parametrize("M,N,K,sk,tile", [
    (1, 6144, 4096, 2, 128), (64, 6144, 4096, 2, 128), (128, 6144, 4096, 2, 128),   # short GEMMs: 96 CTAs
    (4, 4096, 4096, 2, 128),      # 64 CTAs: 6.79 us against 7.25 at split_k 4
    (4, 8192, 4096, 2, 128),      # 11.1 us against 12.4 at split_k 1 (64 CTAs of 1 MiB)
    (4, 2304, 12288, 4, 128),     # 72 CTAs: 9.67 us against 9.97 on 144 64-column CTAs
    (4, 2048, 8192, 4, 128),      # 7.13 us against 12.2 at split_k 8
    (16, 6144, 32768, 4, 128),    # long K: 61.1 us against 67.1 at split_k 2
    (4, 1024, 16384, 4, 64),      # too few 128-column CTAs; 8.62 us against 14.6 at split_k 8
    (4, 49152, 4096, 1, 64)])
def test_auto_split_is_the_measured_best(L, M, N, K, sk, tile):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, 0)
    assert st == lowm.LOWM_OK and (t["split_k"], t["tile_n"]) == (sk, tile)


@pytest.mark.parametrize("M,N,K,sk", [(4, 2304, 12288, 4), (4, 49152, 4096, 2), (16, 6144, 32768, 4),
                                      (64, 6144, 4096, 1), (4, 6144, 4096, 2)])
def test_cluster_counts_for_the_workloads(L, M, N, K, sk):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    assert st == lowm.LOWM_OK and t["split_k"] == sk and t["tiles"] == -(-N // t["tile_n"])
    assert t["tile_n"] in (64, 128)
    mp = 8 if M <= 8 else 16 if M <= 16 else 32 if M <= 32 else 64
    assert t["m_pad"] == (max(mp, 16) if t["tile_n"] == 128 else mp)
    assert t["ctas"] == t["num_clusters"] * sk
    if t["persistent"]:
        # every cluster gets ceil(tiles / clusters) tiles and none is idle
        per = t["tiles_per_cluster"]
        assert per >= 2 and (per - 1) * t["num_clusters"] < t["tiles"] <= per * t["num_clusters"]
    else:
        assert t["num_clusters"] == t["tiles"] and t["tiles_per_cluster"] == 1


@pytest.mark.parametrize("M,N,K,sk,tile,kbs,stages,alias", [
    # the ring (and mailbox placement) each workload measured fastest with on GB300 (tactic sweeps)
    (4, 6144, 4096, 2, 128, 4, 3, 1),       # 8.90 us; 4 x 2 next to the mailbox 9.53 us
    (64, 6144, 4096, 2, 128, 4, 2, 0),      # reduce-scatter mailbox next to the ring 9.88 us; in the ring 10.66 us
    (128, 6144, 4096, 2, 128, 2, 3, 1),     # 13.2 us; 2 x 2 next to the mailbox 16.4 us
    (4, 2304, 12288, 4, 128, 4, 3, 1),      # 9.67 us; 4 x 2 next to the mailbox 11.06, 2 x 5 12.44 us
    (4, 49152, 4096, 2, 64, 2, 2, 0), (4, 49152, 4096, 1, 64, 4, 2, 0),
    (16, 6144, 32768, 4, 128, 2, 3, 1)])    # 61.1 us, two CTAs per SM; 2 x 2 next to the mailbox 63.2, 4 x 3 64.8 us
def test_ring_matches_the_measured_best(L, M, N, K, sk, tile, kbs, stages, alias):
    # the benchmark's launches carry the W-before-PDL promise
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, sk, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    assert st == lowm.LOWM_OK
    assert (t["tile_n"], t["kb_per_stage"], t["stages"], t["mbox_in_ring"]) == (tile, kbs, stages, alias)


@pytest.mark.parametrize("M,N,K,sk,tile,kbs,stages,alias", [
    # without the W promise (default flags, GB300 sweep): the rings within 160 KiB of W
    (4, 6144, 4096, 2, 128, 4, 2, 0),       # 10.67 us; 4 x 3 in the ring 11.17 us
    (64, 6144, 4096, 2, 128, 4, 2, 0),      # reduce-scatter 11.43 us; 2 x 3 owner-only 12.15 us
    (4, 2304, 12288, 4, 128, 4, 3, 1),      # 768 KiB per CTA: 11.50 us; 4 x 2 next to the mailbox 12.12 us
    (16, 6144, 32768, 4, 128, 2, 3, 1)])    # 61.6 us; 2 x 2 next to the mailbox 63.8 us
def test_ring_without_the_w_promise(L, M, N, K, sk, tile, kbs, stages, alias):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    assert st == lowm.LOWM_OK
    assert (t["tile_n"], t["kb_per_stage"], t["stages"], t["mbox_in_ring"]) == (tile, kbs, stages, alias)


def test_query_with_unknown_flags_is_rejected(L):
    st, t = lowm.lowm_gemm_query_tactic_ex(4, 6144, 4096, 2, 4)
    assert st == lowm.LOWM_ERR_INVALID_ARGUMENT and t is None


def test_64_column_rings_with_several_ctas_per_sm_stay_capped(L, monkeypatch):
    # Grids with several CTAs per SM keep at most 160 KiB of W per ring
    # (the one-wave M4 N6144 K4096 ring on 64 columns is 4 x 3 = 96 KiB).
    monkeypatch.setenv("LOWM_TILE_N", "64")
    st, t = lowm.lowm_gemm_query_tactic(4, 6144, 4096, 2)
    assert st == lowm.LOWM_OK and (t["tile_n"], t["kb_per_stage"], t["stages"]) == (64, 4, 3)
    assert t["kb_per_stage"] * t["stages"] * 64 * 64 * 2 <= 160 * 1024


@pytest.mark.parametrize("M,N,K,sk", [(4, 256, 64 * 3, 1), (4, 256, 64 * 6, 1), (4, 256, 64 * 5, 1),
                                      (64, 256, 1024, 8), (64, 6144, 4096, 8), (16, 256, 32768, 4),
                                      (33, 64, 64 * 14, 2), (64, 192, 1024, 8)])
def test_kb_per_stage_divides_the_rank_and_fits(L, M, N, K, sk):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    assert st == lowm.LOWM_OK
    kbr = K // (sk * 64)
    assert kbr % t["kb_per_stage"] == 0
    assert t["smem_bytes"] <= 232448 and t["stages"] >= 2


def test_kb_per_stage_override(L, monkeypatch):
    monkeypatch.setenv("LOWM_KB_PER_STAGE", "8")
    st, t = lowm.lowm_gemm_query_tactic(4, 6144, 4096, 2)
    assert st == lowm.LOWM_OK and t["kb_per_stage"] == 8
    monkeypatch.setenv("LOWM_KB_PER_STAGE", "8")
    st, t = lowm.lowm_gemm_query_tactic(4, 6144, 64 * 6, 1)      # 6 blocks: 8 does not divide, default 2
    assert st == lowm.LOWM_OK and t["kb_per_stage"] == 2


def test_persistent_override_and_cap(L, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", "64")
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", "4")
    st, t = lowm.lowm_gemm_query_tactic(4, 13 * 64, 1024, 2)
    assert st == lowm.LOWM_OK and t["persistent"] == 1
    assert t["num_clusters"] == 4 and t["tiles_per_cluster"] == 4 and t["ctas"] == 8
    monkeypatch.setenv("LOWM_PERSISTENT", "0")
    st, t = lowm.lowm_gemm_query_tactic(4, 49152, 4096, 2)
    assert st == lowm.LOWM_OK and t["persistent"] == 0 and t["ctas"] == 1536


@pytest.mark.parametrize("M,N,K,sk", [(4, 1, 256, 1), (4, 72, 1024, 2), (16, 6150, 1024, 2), (1, 4095, 256, 1),
                                      (64, 136, 1024, 2)])
def test_any_n_is_tiled_with_a_partial_last_tile(L, M, N, K, sk):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    assert st == lowm.LOWM_OK
    tn = t["tile_n"]
    assert t["tiles"] == -(-N // tn) and (t["tiles"] - 1) * tn < N <= t["tiles"] * tn
    if N % 128:
        assert tn == 64          # 128-column tiles only where they divide N (unless forced)


@pytest.mark.parametrize("M,N,K,sk,wpf", [
    # one W stage ahead of the PDL wait for three-stage 64-column rings on a grid that overflows
    # the SMs, the whole ring otherwise (GB300 sweeps)
    (4, 6152, 4096, 2, 1), (4, 6144, 4096, 2, 3), (8, 6144, 4096, 2, 3), (4, 2304, 12288, 4, 3), (4, 49152, 4096, 2, 2),
    (16, 6144, 32768, 4, 3), (64, 6144, 4096, 2, 2), (32, 6144, 4096, 2, 2)])
def test_two_mma_issuers_and_prefetch_depth(L, M, N, K, sk, wpf):
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, sk, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    assert st == lowm.LOWM_OK and t["mma_issuers"] == 2 and t["persistent"] == 0
    assert t["w_prefetch_stages"] == wpf <= t["stages"]


def test_prefetch_depth_override_is_capped_by_the_ring(L, monkeypatch):
    flags = lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT
    monkeypatch.setenv("LOWM_W_PREFETCH", "9")
    st, t = lowm.lowm_gemm_query_tactic_ex(4, 6144, 4096, 2, flags)
    assert st == lowm.LOWM_OK and t["w_prefetch_stages"] == t["stages"]
    monkeypatch.setenv("LOWM_W_PREFETCH", "0")
    st, t = lowm.lowm_gemm_query_tactic_ex(4, 6144, 4096, 2, flags)
    assert st == lowm.LOWM_OK and t["w_prefetch_stages"] == 0


def test_nothing_is_prefetched_before_the_wait_without_the_flag(L):
    # Without LOWM_FLAG_W_BEFORE_PDL_WAIT the kernel requests nothing before
    # griddepcontrol.wait, and the tactic says so.
    for shape in [(4, 6144, 4096, 2), (4, 2304, 12288, 4), (4, 49152, 4096, 2)]:
        st, t = lowm.lowm_gemm_query_tactic(*shape)
        assert st == lowm.LOWM_OK and t["w_prefetch_stages"] == 0


@pytest.mark.parametrize("M,N,K,sk,flags,l2bw", [
    # GB300, default flags: one stage of W into L2 before the wait for short streams (M4 N6144 K4096 10.60 ->
    # 10.25 us), the whole ring for long ones (M4 N2304 K12288 split_k 4 11.69 -> 11.25 us); none with the
    # W promise, which requests the ring itself before the wait
    (4, 6144, 4096, 2, 0, 1), (64, 6144, 4096, 0, 0, 1), (4, 2304, 12288, 4, 0, 3), (16, 6144, 32768, 4, 0, 3),
    (4, 6144, 4096, 2, 1, 0), (4, 2304, 12288, 4, 1, 0)])
def test_l2_requests_before_the_wait(L, M, N, K, sk, flags, l2bw):
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, sk, flags)
    assert st == lowm.LOWM_OK and t["l2_before_wait_stages"] == l2bw


def test_persistent_schedule_has_one_issuer(L, monkeypatch):
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    st, t = lowm.lowm_gemm_query_tactic(4, 49152, 4096, 2)
    assert st == lowm.LOWM_OK
    if t["persistent"]:
        assert t["mma_issuers"] == 1


@pytest.mark.parametrize("M,m_pad", [(65, 96), (96, 96), (97, 128), (127, 128), (128, 128)])
def test_m_up_to_128_pads_to_96_or_128(L, M, m_pad, monkeypatch):
    monkeypatch.setenv("LOWM_PERSISTENT", "1")      # no persistent m_pad 96 / 128 instance: ignored
    for sk in (1, 2, 3, 4):
        st, t = lowm.lowm_gemm_query_tactic(M, 6144, 4096, sk)
        assert st == lowm.LOWM_OK and t["m_pad"] == m_pad and t["persistent"] == 0 and t["mma_issuers"] == 2
        assert t["smem_bytes"] <= 232448
        assert t["mbox_in_ring"] == (1 if sk > 1 else 0)       # the 24-64 KiB slots share the drained ring
    st, t = lowm.lowm_gemm_query_tactic(M, 64, 8192, 0)   # one tile: auto split stops where the mailbox fits
    assert st == lowm.LOWM_OK and t["split_k"] == 4


def test_forced_128_column_tiles_at_m_pad_128(L, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", "128")
    st, t = lowm.lowm_gemm_query_tactic(128, 6144, 4096, 2)
    assert st == lowm.LOWM_OK and t["tile_n"] == 128 and t["m_pad"] == 128
    st, t = lowm.lowm_gemm_query_tactic(128, 6144, 4096, 4)    # no 128-column split-4 instance: 64 columns
    assert st == lowm.LOWM_OK and t["tile_n"] == 64


def test_auto_split_k_keeps_the_k_loop_non_empty(L):
    for M, N, K in [(4, 64, 64), (4, 64, 128), (4, 6144, 4096), (64, 64, 512), (1, 49152, 4096)]:
        st, t = lowm.lowm_gemm_query_tactic(M, N, K, 0)
        assert st == lowm.LOWM_OK
        assert K % (t["split_k"] * 64) == 0 and K // (t["split_k"] * 64) >= 1


@pytest.mark.parametrize("M,N,K,sk,want", [
    (0, 64, 64, 1, lowm.LOWM_ERR_INVALID_ARGUMENT),
    (129, 64, 64, 1, lowm.LOWM_ERR_UNSUPPORTED_SHAPE),
    (128, 64, 1024, 8, lowm.LOWM_ERR_UNSUPPORTED_SHAPE),   # m_pad 128: the split-8 mailbox does not fit
    (4, 64, 96, 1, lowm.LOWM_ERR_UNSUPPORTED_SHAPE),      # K not a multiple of 64
    (4, 64, 64, 2, lowm.LOWM_ERR_UNSUPPORTED_SHAPE),      # empty K loop on one rank
    (4, 64, 128, 3, lowm.LOWM_ERR_UNSUPPORTED_SHAPE),     # 2 K blocks for 3 ranks: an empty share
    (4, 64, 128, 5, lowm.LOWM_ERR_INVALID_ARGUMENT),      # split_k outside {0, 1, 2, 3, 4, 8}
    (4, 64, 64 * 5, 6, lowm.LOWM_ERR_INVALID_ARGUMENT),
    (4, 64, 1024, 16, lowm.LOWM_ERR_INVALID_ARGUMENT),
    (4, -64, 64, 1, lowm.LOWM_ERR_INVALID_ARGUMENT),
])
def test_query_rejects_bad_shapes(L, M, N, K, sk, want):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    assert st == want and t is None


def test_gemm_rejects_null_and_misaligned_pointers_before_touching_a_device(L):
    assert lowm.lowm_gemm_bf16(0, 0x1000, 0x2000, 4, 64, 64, 1, 0) == lowm.LOWM_ERR_INVALID_ARGUMENT
    assert lowm.lowm_gemm_bf16(0x1000, 0x2000, 0x3008, 4, 64, 64, 1, 0) == lowm.LOWM_ERR_MISALIGNED
    assert lowm.lowm_gemm_bf16(0x1000, 0x2000, 0x3000, 0, 64, 64, 1, 0) == lowm.LOWM_ERR_INVALID_ARGUMENT
    # C overlapping W
    assert lowm.lowm_gemm_bf16(0x1000, 0x100000, 0x100040, 4, 64, 64, 1, 0) == lowm.LOWM_ERR_INVALID_ARGUMENT
    assert lowm.lowm_gemm_bf16_debug(0x1000, 0x100000, 0x200000, 4, 64, 64, 1, 0, stages=1) \
        == lowm.LOWM_ERR_INVALID_ARGUMENT
    assert lowm.lowm_gemm_bf16_host(0, 1, 1, 1, 1, 1, 4, 64, 64, 0, 0) == lowm.LOWM_ERR_INVALID_ARGUMENT
    assert lowm.lowm_tmem_hog_launch(0, 1, 48, 1) == lowm.LOWM_ERR_INVALID_ARGUMENT
    assert lowm.lowm_gemm_bf16_ex(0x1000, 0x100000, 0x200000, 4, 64, 64, 1, 4, 0) == lowm.LOWM_ERR_INVALID_ARGUMENT


def test_library_does_not_reference_the_oracle():
    src_dir = os.path.join(ROOT, "split_bf16_gemm_swap_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle." not in text, f


C_PROGRAM = r"""
#include <stdio.h>
#include "lowm_gemm.h"

int main(void)
{
    lowm_tactic_t t;
    lowm_status_t st = lowm_gemm_query_tactic(4, 6144, 4096, 2, &t);
    if (st != LOWM_OK) { printf("query failed: %s\n", lowm_status_string(st)); return 1; }
    printf("%d %d %d %d %d %d %d %d\n", t.tile_n, t.m_pad, t.split_k, t.kb_per_stage, t.stages, t.ctas,
           t.mma_issuers, t.w_prefetch_stages);
    if (lowm_gemm_query_tactic(129, 64, 64, 1, &t) != LOWM_ERR_UNSUPPORTED_SHAPE) return 2;
    if (lowm_gemm_bf16(0, 0, 0, 4, 64, 64, 1, 0) != LOWM_ERR_INVALID_ARGUMENT) return 3;
    if (lowm_gemm_bf16_ex((void *)0x1000, (void *)0x2000, (void *)0x3000, 4, 64, 64, 1, 4u, 0)
        != LOWM_ERR_INVALID_ARGUMENT) return 4;      /* unknown flag bit */
    return 0;
}
"""


def test_the_header_is_c99_and_links_against_the_library(L, tmp_path):
    # The boundary from plain C: the header compiles as C99, the program links
    # against liblowm_gemm.so and the host-only entry points answer as the
    # Python binding does.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lowm.LIB_PATH)
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-L", libdir, "-llowm_gemm", "-Wl,-rpath," + libdir, "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    st, t = lowm.lowm_gemm_query_tactic(4, 6144, 4096, 2)
    want = [t[k] for k in ("tile_n", "m_pad", "split_k", "kb_per_stage", "stages", "ctas", "mma_issuers",
                           "w_prefetch_stages")]
    assert [int(x) for x in out.stdout.split()] == want


@pytest.mark.parametrize("M,kbs,stages", [(80, 4, 2), (96, 4, 2), (128, 2, 3)])
def test_m_pad_96_and_128_tactics_are_the_measured_best(L, M, kbs, stages):
    # GB300 sweeps at N6144 K4096: 128-column tiles, split_k 2, the mailbox in
    # the drained ring.  m_pad 128: 2 x 3 ring, 14.1 us against 15.8 us for
    # split_k 1 on 64-column tiles and 15.8-18.2 us for other rings.  m_pad 96:
    # 4 x 2 ring, M96 11.84 us (12.97 us on m_pad 128), against 12.30 for 2 x
    # 3 or 2 x 4 and 16.7 for 1 x 6.
    st, t = lowm.lowm_gemm_query_tactic(M, 6144, 4096, 0)
    assert st == lowm.LOWM_OK
    assert (t["tile_n"], t["split_k"], t["kb_per_stage"], t["stages"], t["ctas"], t["mbox_in_ring"]) == \
        (128, 2, kbs, stages, 96, 1)


@pytest.mark.parametrize("K,sk", [(64 * 3, 2), (64 * 7, 3), (4096, 3), (64 * 50, 3), (64 * 9, 4)])
def test_uneven_k_shares_are_accepted(L, K, sk):
    # K is cut into whole stages; ranks whose share would be uneven take one
    # stage fewer than the last ones, and every rank keeps at least one stage.
    st, t = lowm.lowm_gemm_query_tactic(4, 640, K, sk)
    assert st == lowm.LOWM_OK and t["split_k"] == sk
    total = K // 64 // t["kb_per_stage"]
    assert (K // 64) % t["kb_per_stage"] == 0 and total >= sk
    shares = [(r + 1) * total // sk - r * total // sk for r in range(sk)]
    assert min(shares) >= 1 and max(shares) - min(shares) <= 1 and sum(shares) == total


def test_split3_defaults_to_the_mailbox_in_the_ring(L, monkeypatch):
    st, t = lowm.lowm_gemm_query_tactic(64, 6144, 4096, 3)
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == 1
    st, t = lowm.lowm_gemm_query_tactic(4, 6152, 4096, 2)       # a mailbox of 2 KiB: no larger ring to gain
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == 0
    st, t = lowm.lowm_gemm_query_tactic_ex(4, 6144, 4096, 2, 1)  # sharing the ring makes room for a third stage
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == 1 and t["stages"] == 3
    monkeypatch.setenv("LOWM_MBOX_IN_RING", "0")
    st, t = lowm.lowm_gemm_query_tactic(4, 640, 64 * 9, 3)
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == 0
    st, t = lowm.lowm_gemm_query_tactic(4, 640, 64 * 9, 1)
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == 0          # no mailbox at split_k 1


def test_every_tactic_of_a_shape_grid_is_launchable(L):
    # Over a grid of shapes, splits and both launch flags, every accepted
    # tactic fits the SM, tiles K in whole stages and reports consistent
    # counts; the host refuses exactly the documented rest (fewer K blocks
    # than ranks, M above 64 with split_k 8) before any launch.
    for M in (1, 3, 4, 8, 16, 17, 32, 33, 64, 65, 96, 128):
        for N in (1, 63, 64, 200, 1024, 2304, 4096, 6144, 6152, 49152):
            for K in (64, 1024, 4096, 12288, 32768):
                for sk in (0, 1, 2, 3, 4, 8):
                    for flags in (0, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT):
                        st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, sk, flags)
                        refuse = K // 64 < max(sk, 1) or (M > 64 and sk == 8)
                        assert (st == lowm.LOWM_ERR_UNSUPPORTED_SHAPE) == refuse, (M, N, K, sk, flags, st)
                        if refuse:
                            continue
                        where = (M, N, K, sk, flags, t)
                        assert t["smem_bytes"] <= 232448 and t["stages"] >= 2, where
                        assert (K // 64) % t["kb_per_stage"] == 0 and K // (64 * t["kb_per_stage"]) >= t["split_k"], where
                        assert t["tile_n"] in (64, 128) and (t["tile_n"] == 64 or N % 128 == 0), where
                        assert t["m_pad"] >= M and t["tiles"] == -(-N // t["tile_n"]), where
                        assert t["ctas"] == t["num_clusters"] * t["split_k"] and (sk == 0 or t["split_k"] == sk), where
                        assert 0 <= t["w_prefetch_stages"] <= t["stages"], where
                        if flags:
                            assert t["l2_before_wait_stages"] == 0, where
                        else:
                            assert t["w_prefetch_stages"] == 0 and 0 <= t["l2_before_wait_stages"] <= t["stages"], where
