"""Race stress of the TMEM release ordering, on the GPU.

The method of the TensorRT-LLM PR "Fix two synchronization gaps in the
MiniMax M3 low-M split-K GEMM" (Hardware verification): stall two of the four
epilogue warps before their first arrival on the TMEM barrier (5, 10 and
100 us), keep the shared-memory request at the kernel's footprint so another
kernel can co-reside on the SM, run a kernel on a second stream that
allocates TMEM columns, fills them with NaN and frees them, and probe
%globaltimer at the epilogue's tcgen05.ld and at the MMA warp's
tcgen05.dealloc.  20 launches per configuration.

Pass criteria: every stressed output is bitwise identical to the unstressed
output (which is itself checked against the oracle / the closed form), no
kernel wait times out, and in every CTA the MMA warp saw all four epilogue
warps' ordering tickets just before tcgen05.dealloc (each ticket is taken
after that warp's last tcgen05.wait::ld), with the dealloc timestamp not
earlier than the latest epilogue load as a second, clock-based check.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_parity
from split_bf16_gemm_swap_gb300 import build, inputs, lowm

pytestmark = pytest.mark.gpu

DEV = "cuda"
LAUNCHES = 20
STALL_WARPS = (1 << 4) | (1 << 5)          # two of the four epilogue warps (2..5)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    lowm.lib()


def stressed(Ad, Wd, M, N, K, split_k, stall_ns, hog_cols=256, stall_rank_mask=0, warp_mask=STALL_WARPS, flags=0):
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, split_k, flags)
    assert st == lowm.LOWM_OK
    ctas = t["ctas"]
    s_gemm = torch.cuda.Stream()
    s_hog = torch.cuda.Stream()
    probes = torch.zeros((LAUNCHES, ctas, 3), dtype=torch.int64, device=DEV)
    outs = torch.empty((LAUNCHES, M, N), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    for i in range(LAUNCHES):
        for _ in range(3):
            assert lowm.lowm_tmem_hog_launch(s_hog, 4096, hog_cols, 4) == lowm.LOWM_OK
        st = lowm.lowm_gemm_bf16_debug(Ad, Wd, outs[i], M, N, K, split_k, s_gemm, stall_warp_mask=warp_mask,
                                       stall_rank_mask=stall_rank_mask, stall_ns=stall_ns, probes=probes[i],
                                       flags=flags)
        assert st == lowm.LOWM_OK
    torch.cuda.synchronize()
    st, detail = lowm.lowm_gemm_sync_status(s_gemm)
    assert st == lowm.LOWM_OK, "kernel wait timed out, bits %#x" % detail
    return outs, probes.cpu().numpy()


EPILOGUE_WARPS = 4


def check_probes(p):
    t_ld, t_dealloc, tickets = p[..., 0], p[..., 1], p[..., 2]
    assert np.all(t_ld > 0) and np.all(t_dealloc > 0), "a CTA did not record both probes"
    short = int(np.sum(tickets != EPILOGUE_WARPS))
    assert short == 0, "%d of %d CTAs freed TMEM without all %d epilogue warps' tickets (seen: %s)" % (
        short, tickets.size, EPILOGUE_WARPS, sorted(set(tickets.ravel().tolist())))
    early = int(np.sum(t_dealloc < t_ld))
    assert early == 0, "%d of %d CTAs freed TMEM before the epilogue's last load" % (early, t_ld.size)


CONFIGS = [
    # M, N, K, split_k, kind
    (16, 6144, 32768, 4, "int"),
    (4, 6144, 4096, 2, "randn"),
    (4, 2304, 12288, 4, "randn"),
    (4, 49152, 4096, 2, "randn"),
    (64, 6144, 4096, 2, "randn"),          # 128-column tiles (MMA M = 128)
    (128, 6144, 4096, 2, "randn"),         # m_pad 128: chunked epilogue, release after the last chunk
    (64, 6144, 4096, 3, "randn"),          # split_k 3: uneven K shares, mailbox in the drained ring
    (128, 6144, 4096, 3, "randn"),
    (16, 6144, 32768, 3, "int"),
]


@pytest.mark.parametrize("M,N,K,split_k,kind", CONFIGS)
def test_stalled_epilogue_with_tmem_hog(M, N, K, split_k, kind):
    A, W = inputs.make_problem(M, N, K, seed=1234, kind=kind)
    Ad, Wd = A.to(DEV), W.to(DEV)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    F = torch.empty((M, N), dtype=torch.float32, device=DEV)
    assert lowm.lowm_gemm_bf16_debug(Ad, Wd, ref, M, N, K, split_k, None, c_f32=F) == lowm.LOWM_OK
    torch.cuda.synchronize()
    ref_bits = inputs.bits(ref.cpu())
    if kind == "int":
        col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
        assert np.array_equal(ref_bits, np.broadcast_to(inputs.bits(col[None, :]), ref_bits.shape))
    else:
        Cref, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
        assert_parity(ref_bits, F.cpu().numpy().astype(np.float64), Cref, S, A, W)
    for stall_ns in (5_000, 10_000, 100_000):
        outs, probes = stressed(Ad, Wd, M, N, K, split_k, stall_ns)
        o = outs.view(torch.int16)
        bad = int((o != ref.view(torch.int16)[None]).any(dim=2).any(dim=1).sum())
        assert bad == 0, "stall %d ns: %d of %d launches differ from the unstressed output" % (
            stall_ns, bad, LAUNCHES)
        check_probes(probes)


@pytest.mark.parametrize("M,N,K,split_k", [(4, 6144, 4096, 2), (16, 6144, 32768, 4), (128, 1024, 4096, 2)])
def test_stalled_second_mma_issuer_with_tmem_hog(M, N, K, split_k):
    # The columns may be freed only after both issuers' final commits: delay
    # the second issuer (warp 6) before its first MMA, with the TMEM hog on a
    # second stream; outputs must stay bitwise identical and every CTA's
    # dealloc must follow its epilogue's last load.
    A, W = inputs.make_problem(M, N, K, seed=1234, kind="int")
    Ad, Wd = A.to(DEV), W.to(DEV)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16(Ad, Wd, ref, M, N, K, split_k, None) == lowm.LOWM_OK
    torch.cuda.synchronize()
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(inputs.bits(ref.cpu()), np.broadcast_to(inputs.bits(col[None, :]), (M, N)))
    for stall_ns in (5_000, 100_000):
        outs, probes = stressed(Ad, Wd, M, N, K, split_k, stall_ns, warp_mask=1 << 6)
        assert bool((outs.view(torch.int16) == ref.view(torch.int16)[None]).all())
        check_probes(probes)


@pytest.mark.parametrize("M,stall_rank_mask", [(4, 1), (4, 2), (64, 1), (64, 2)])
def test_stalling_only_one_rank(M, stall_rank_mask):
    # The pages also stall only the owner or only the non-owner rank.  At M64
    # (reduce-scatter) each rank is both sender and receiver.
    N, K, split_k = 6144, 4096, 2
    A, W = inputs.make_problem(M, N, K, seed=77)
    Ad, Wd = A.to(DEV), W.to(DEV)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16(Ad, Wd, ref, M, N, K, split_k, None) == lowm.LOWM_OK
    outs, probes = stressed(Ad, Wd, M, N, K, split_k, 10_000, hog_cols=32, stall_rank_mask=stall_rank_mask)
    assert bool((outs.view(torch.int16) == ref.view(torch.int16)[None]).all())
    check_probes(probes)


@pytest.mark.parametrize("tile", ["64", "128"])
def test_persistent_schedule_under_stress(tile, monkeypatch):
    # Several tiles per cluster: the TMEM release after the last tile and the
    # double-buffered mailbox hand-off, under the same stall + hog method.
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", "16")
    monkeypatch.setenv("LOWM_TILE_N", tile)
    M, N, K, split_k = 16, 6144, 8192, 2
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK and t["persistent"] == 1 and t["tiles_per_cluster"] >= 3
    A, W = inputs.make_problem(M, N, K, seed=1234, kind="int")
    Ad, Wd = A.to(DEV), W.to(DEV)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16(Ad, Wd, ref, M, N, K, split_k, None) == lowm.LOWM_OK
    torch.cuda.synchronize()
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(inputs.bits(ref.cpu()), np.broadcast_to(inputs.bits(col[None, :]), (M, N)))
    outs, probes = stressed(Ad, Wd, M, N, K, split_k, 10_000)
    assert bool((outs.view(torch.int16) == ref.view(torch.int16)[None]).all())
    check_probes(probes)


@pytest.mark.parametrize("M,N,K,split_k", [(4, 6144, 4096, 2), (64, 6144, 4096, 2), (16, 6144, 32768, 4)])
def test_stress_with_the_w_promise(M, N, K, split_k):
    # The timed tactics (LOWM_FLAG_W_BEFORE_PDL_WAIT: the deeper rings, W
    # requested before the dependency wait; at M4 the mailbox in the ring, at
    # M64 the reduce-scatter exchange) under the same stall + TMEM hog method.
    flags = lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, split_k, flags)
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == (0 if M == 64 else 1)
    A, W = inputs.make_problem(M, N, K, seed=1234, kind="int")
    Ad, Wd = A.to(DEV), W.to(DEV)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16_ex(Ad, Wd, ref, M, N, K, split_k, flags, None) == lowm.LOWM_OK
    torch.cuda.synchronize()
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(inputs.bits(ref.cpu()), np.broadcast_to(inputs.bits(col[None, :]), (M, N)))
    for stall_ns in (5_000, 100_000):
        outs, probes = stressed(Ad, Wd, M, N, K, split_k, stall_ns, flags=flags)
        assert bool((outs.view(torch.int16) == ref.view(torch.int16)[None]).all())
        check_probes(probes)


SOAK_CONFIGS = [  # M, N, K, split_k, flags
    (4, 6144, 4096, 2, 1), (4, 6144, 4096, 2, 0), (64, 6144, 4096, 2, 1), (96, 6144, 4096, 2, 1),
    (128, 6144, 4096, 2, 1), (4, 2304, 12288, 4, 1), (16, 6144, 32768, 4, 1), (64, 6144, 4096, 3, 0),
    (4, 49152, 4096, 2, 1), (32, 4096, 4096, 0, 1)]


@pytest.mark.parametrize("M,N,K,split_k,flags", SOAK_CONFIGS)
def test_soak(M, N, K, split_k, flags):
    # The extended soak: LOWM_SOAK_ROUNDS rounds (unset: skipped) of the four
    # stall patterns (warps 4 and 5, the second issuer, or all three; 5 or
    # 50 us) with the TMEM hog, 20 launches each, integer inputs against the
    # closed form.  80 rounds are 6,400 launches per configuration.
    import os
    rounds = int(os.environ.get("LOWM_SOAK_ROUNDS", "0"))
    if rounds <= 0:
        pytest.skip("set LOWM_SOAK_ROUNDS to run the extended soak")
    A, W = inputs.make_problem(M, N, K, seed=4242, kind="int")
    Ad, Wd = A.to(DEV), W.to(DEV)
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    want = np.broadcast_to(inputs.bits(col[None, :]), (M, N))
    stalls = [(STALL_WARPS, 5_000), (STALL_WARPS, 50_000), (1 << 6, 5_000), (STALL_WARPS | (1 << 6), 50_000)]
    differing = 0
    for _ in range(rounds):
        for warp_mask, stall_ns in stalls:
            outs, probes = stressed(Ad, Wd, M, N, K, split_k, stall_ns, warp_mask=warp_mask, flags=flags)
            differing += int((inputs.bits(outs.cpu()) != want[None]).any(axis=(1, 2)).sum())
            check_probes(probes)
    assert differing == 0, "%d of %d launches differ from the closed form" % (differing, rounds * len(stalls) * LAUNCHES)
