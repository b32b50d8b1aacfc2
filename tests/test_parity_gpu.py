"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar (from the method's own check, "Fix two synchronization gaps in the
MiniMax M3 low-M split-K GEMM", Hardware verification, which compares the bf16
output with an fp32 product, and the exact-integer construction of
"warpgroup_mma_wait does not properly synchronize across warpgroups"):
  * integer-valued inputs: bit-exact, fp32 sums included;
  * random inputs: the kernel's fp32 sums within 1e-5 * sqrt(K) * max|a| *
    max|w| of the oracle's fp64 sums, the bf16 output exactly the
    round-to-nearest-even of those fp32 sums, and within 1 bf16 ulp of the
    oracle's single-rounded value wherever that bound is below a quarter ulp
    (for outputs that cancel to a few ulps of the fp32 error, the absolute
    bound is the bar, as it is for any fp32-accumulating GEMM);
  * repeated launches: bitwise identical.
Every case compares every output element.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    lowm.lib()
    torch.cuda.init()


def sync_ok():
    st, detail = lowm.lowm_gemm_sync_status()
    assert st == lowm.LOWM_OK, "kernel status %d, bits %#x" % (st, detail)


def run_gpu(A, W, split_k=0, want_f32=True, **dbg):
    M, K = A.shape
    N = W.shape[0]
    Ad, Wd = A.to(DEV), W.to(DEV)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)   # unwritten outputs stay NaN
    F = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV) if want_f32 else None
    st = lowm.lowm_gemm_bf16_debug(Ad, Wd, C, M, N, K, split_k, None, c_f32=F, **dbg)
    assert st == lowm.LOWM_OK, lowm.status_string(st)
    sync_ok()
    return inputs.bits(C.cpu()), (F.cpu().numpy().astype(np.float64) if F is not None else None)


def check(A, W, split_k=0, exact=False, flags=0):
    M, K = A.shape
    C, F = run_gpu(A, W, split_k, flags=flags)
    Cref, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    if exact:
        bad = np.argwhere(C != Cref)
        assert bad.size == 0, "first mismatches (m, n): %s" % bad[:8].tolist()
        assert np.array_equal(F, S)
        return C
    assert_parity(C, F, Cref, S, A, W, label="M%d N%d K%d split_k %d" % (M, W.shape[0], K, split_k))
    return C


# ---------------------------------------------------------------- small shapes
SMALL = [
    # M, N, K, split_k: several tiles, ragged M, ring wrap-around (K/64 > stages), every m_pad and split_k
    (1, 64, 64, 1), (3, 192, 256, 1), (4, 640, 1024, 2), (5, 128, 512, 4), (8, 64, 1024, 8),
    (7, 256, 4096, 1), (13, 256, 1024, 2), (16, 128, 2048, 4), (17, 192, 512, 1), (24, 128, 4096, 2),
    (31, 64, 512, 2), (32, 320, 1024, 2), (33, 128, 256, 1), (48, 64, 1024, 4), (64, 192, 1024, 8),
    (64, 128, 8192, 1), (2, 1024, 2048, 0), (9, 448, 3072, 0),
]


@pytest.mark.parametrize("M,N,K,split_k", SMALL)
def test_small_shapes_random(M, N, K, split_k):
    A, W = inputs.make_problem(M, N, K, seed=100 + M + N + K)
    check(A, W, split_k)


@pytest.mark.parametrize("M,N,K,split_k", [(4, 128, 512, 1), (16, 192, 1024, 2), (64, 64, 2048, 4),
                                           (3, 320, 4096, 8)])
def test_small_shapes_integer_exact(M, N, K, split_k):
    A, W = inputs.make_problem(M, N, K, seed=7, kind="int")
    C = check(A, W, split_k, exact=True)
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(C, np.broadcast_to(inputs.bits(col[None, :]), C.shape))


def test_identity_weight_maps_every_column():
    # W[n, k] = 1 iff k == n: C[m, n] = A[m, n] exactly, so a wrong TMEM lane /
    # column mapping or a transposed store shows up as a permutation.
    M, N, K = 8, 64, 128
    A = (torch.arange(M * K, dtype=torch.float32).reshape(M, K) % 251 + 1).to(torch.bfloat16)
    W = torch.zeros((N, K), dtype=torch.bfloat16)
    W[torch.arange(N), torch.arange(N)] = 1.0
    for split_k in (1, 2):
        C, _ = run_gpu(A, W, split_k, want_f32=False)
        want = inputs.bits(A)[:, :N]
        if not np.array_equal(C, want):
            vals = {int(v): i for i, v in enumerate(want[0])}
            got_cols = [vals.get(int(v), -1) for v in C[0]]
            raise AssertionError("split_k %d: output column n holds input column %s" % (split_k, got_cols))


def test_rows_beyond_M_are_not_written():
    M, N, K = 3, 256, 512
    A, W = inputs.make_problem(M, N, K, seed=3)
    big = torch.full((M + 5, N), 7.0, dtype=torch.bfloat16, device=DEV)
    F = torch.empty((M, N), dtype=torch.float32, device=DEV)
    st = lowm.lowm_gemm_bf16_debug(A.to(DEV), W.to(DEV), big, M, N, K, 2, None, c_f32=F)
    assert st == lowm.LOWM_OK
    sync_ok()
    assert torch.all(big[M:] == 7.0)
    Cref, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert_parity(inputs.bits(big[:M].cpu()), F.cpu().numpy().astype(np.float64), Cref, S, A, W)


# ---------------------------------------------------------------- the five workloads at full size
def test_workload_m4_n6144_k4096_split2():
    A, W = inputs.make_problem(4, 6144, 4096, seed=1234)
    check(A, W, 2)


def test_workload_m4_n2304_k12288_split4():
    A, W = inputs.make_problem(4, 2304, 12288, seed=1234)
    check(A, W, 4)


def test_workload_m4_n49152_k4096_split2():
    A, W = inputs.make_problem(4, 49152, 4096, seed=1234)
    check(A, W, 2)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64, 96, 128])
def test_workload_m_sweep_n6144_k4096(M):
    A, W = inputs.make_problem(M, 6144, 4096, seed=1234)
    st, t = lowm.lowm_gemm_query_tactic(M, 6144, 4096, 0)
    assert st == lowm.LOWM_OK and t["split_k"] in (1, 2, 4)
    check(A, W, 0)


def test_workload_integer_m16_n6144_k32768_split4():
    A, W = inputs.make_problem(16, 6144, 32768, seed=1234, kind="int")
    C = check(A, W, 4, exact=True)
    col = W.to(torch.int64).sum(dim=1)
    assert int(col.abs().max()) < 2 ** 24
    want = inputs.bits(col.to(torch.float32).to(torch.bfloat16)[None, :])
    assert np.array_equal(C, np.broadcast_to(want, C.shape))


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("M,N,K,split_k", [(4, 6144, 4096, 2), (4, 2304, 12288, 4), (16, 6144, 32768, 4)])
def test_twenty_launches_are_bitwise_identical(M, N, K, split_k):
    A, W = inputs.make_problem(M, N, K, seed=99)
    Ad, Wd = A.to(DEV), W.to(DEV)
    outs = torch.empty((20, M, N), dtype=torch.bfloat16, device=DEV)
    for i in range(20):
        assert lowm.lowm_gemm_bf16(Ad, Wd, outs[i], M, N, K, split_k, None) == lowm.LOWM_OK
    sync_ok()
    o = outs.view(torch.int16)
    assert bool((o == o[0:1]).all())


def test_every_split_k_agrees_with_the_oracle():
    A, W = inputs.make_problem(4, 1024, 8192, seed=5)
    for sk in (1, 2, 4, 8):
        check(A, W, sk)


def test_pdl_chain_reads_the_previous_output():
    # Each GEMM's A is the previous GEMM's C, launched back to back with PDL:
    # griddepcontrol.wait must order the TMA reads of A after the producer's stores.
    M, D = 4, 1024
    A0, _ = inputs.make_problem(M, D, D, seed=11)
    Ws = [inputs.make_problem(M, D, D, seed=20 + i)[1] for i in range(6)]
    Wd = [w.to(DEV) for w in Ws]
    Cs = [A0.to(DEV)] + [torch.empty((M, D), dtype=torch.bfloat16, device=DEV) for _ in Ws]
    Fs = [torch.empty((M, D), dtype=torch.float32, device=DEV) for _ in Ws]
    for i, w in enumerate(Wd):
        assert lowm.lowm_gemm_bf16_debug(Cs[i], w, Cs[i + 1], M, D, D, 2, None, c_f32=Fs[i]) == lowm.LOWM_OK
    sync_ok()
    for i, w in enumerate(Ws):
        a = Cs[i].cpu()
        ref, S = oracle.gemm_bf16_f64(inputs.bits(a), inputs.bits(w))
        assert_parity(inputs.bits(Cs[i + 1].cpu()), Fs[i].cpu().numpy().astype(np.float64), ref, S, a, w)


def test_host_buffer_entry_point_matches_device_path():
    M, N, K = 4, 6144, 4096
    A, W = inputs.make_problem(M, N, K, seed=1234)
    Ah, Wh = A.pin_memory(), W.pin_memory()
    Ch = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    Ad = torch.empty_like(A, device=DEV)
    Wd = torch.empty_like(W, device=DEV)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16_host(Ah, Wh, Ch, Ad, Wd, Cd, M, N, K, 2, None) == lowm.LOWM_OK
    C_dev, _ = run_gpu(A, W, 2, want_f32=False)
    assert np.array_equal(inputs.bits(Ch), C_dev)


def test_shipped_tactic_with_full_capacity_request_gives_the_same_bits(monkeypatch):
    # The pages' shipped tactic: 10 stages of one 64-wide K block, full-capacity
    # shared-memory request (nothing else can co-reside on the SM).
    A, W = inputs.make_problem(4, 6144, 4096, seed=8)
    C1, _ = run_gpu(A, W, 2, want_f32=False)
    monkeypatch.setenv("LOWM_KB_PER_STAGE", "1")
    C2, _ = run_gpu(A, W, 2, want_f32=False, full_smem=1, stages=10)
    assert np.array_equal(C1, C2)


def test_a_dropped_mailbox_times_out_and_the_context_survives():
    # Failure injection on the host side of the protocol: the non-owner ranks
    # skip their publication, so the owner's bounded mailbox wait runs out.
    A, W = inputs.make_problem(4, 256, 1024, seed=4)
    Ad, Wd = A.to(DEV), W.to(DEV)
    C = torch.empty((4, 256), dtype=torch.bfloat16, device=DEV)
    st = lowm.lowm_gemm_bf16_debug(Ad, Wd, C, 4, 256, 1024, 2, None, drop_mailbox=1,
                                   reduce_timeout_ns=20_000_000)
    assert st == lowm.LOWM_OK
    st, detail = lowm.lowm_gemm_sync_status()
    assert st == lowm.LOWM_ERR_TIMEOUT and detail == (1 << 8), (st, hex(detail))
    # the status word was cleared and the context still works
    check(A, W, 2)


@pytest.mark.parametrize("M,split_k", [(64, 2), (64, 4), (32, 2)])
def test_a_dropped_two_phase_mailbox_times_out(M, split_k):
    # m_pad 64 with split_k 4 waits on two mailbox halves, m_pad 32 on one,
    # and m_pad 64 with split_k 2 (reduce-scatter) on one per rank, every rank
    # a receiver; every bounded wait must run out, report the mailbox bit,
    # and leave a working context.
    N, K = 256, 1024
    A, W = inputs.make_problem(M, N, K, seed=5)
    Ad, Wd = A.to(DEV), W.to(DEV)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    st = lowm.lowm_gemm_bf16_debug(Ad, Wd, C, M, N, K, split_k, None, drop_mailbox=1,
                                   reduce_timeout_ns=20_000_000)
    assert st == lowm.LOWM_OK
    st, detail = lowm.lowm_gemm_sync_status()
    assert st == lowm.LOWM_ERR_TIMEOUT and detail == (1 << 8), (st, hex(detail))
    check(A, W, split_k)


# ---------------------------------------------------------------- reduce-scatter exchange (m_pad 64, split_k 2)
@pytest.mark.parametrize("M,N,flags", [(33, 6144, 1), (40, 6144, 0), (47, 256, 0), (48, 6144, 1), (63, 200, 0),
                                       (64, 6144, 0), (64, 6144, 1), (64, 6150, 1), (64, 70, 0), (64, 1, 0)])
def test_reduce_scatter_rows(M, N, flags):
    # Each rank keeps half of the 48 or 64 padded rows: rank 1's half holds
    # 1..24 or 1..32 real rows, and 64- and 128-column tiles, N tails and both
    # launch flags take the same exchange.
    K = 4096
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, 2, flags)
    assert st == lowm.LOWM_OK and (t["m_pad"], t["split_k"], t["mbox_in_ring"]) == (48 if M <= 48 else 64, 2, 0)
    A, W = inputs.make_problem(M, N, K, seed=1400 + M + N)
    check(A, W, 2, flags=flags)


def test_reduce_scatter_is_exact_on_integer_inputs():
    # Integer operands: both halves bit-exact in bf16 and in the fp32 sums.
    A, W = inputs.make_problem(64, 6144, 8192, seed=1410, kind="int")
    check(A, W, 2, exact=True)


def test_reduce_scatter_twenty_launches_are_bitwise_identical():
    M, N, K = 64, 6144, 4096
    A, W = inputs.make_problem(M, N, K, seed=1420)
    Ad, Wd = A.to(DEV), W.to(DEV)
    outs = torch.empty((20, M, N), dtype=torch.bfloat16, device=DEV)
    for i in range(20):
        assert lowm.lowm_gemm_bf16_ex(Ad, Wd, outs[i], M, N, K, 2, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT, None) == \
            lowm.LOWM_OK
    sync_ok()
    o = outs.view(torch.int16)
    assert bool((o == o[0:1]).all())


def test_w_before_pdl_wait_flag_keeps_the_chain_correct():
    # W is never written by the preceding kernel here, so the flag's promise holds;
    # A is the previous GEMM's output and must still be read after the wait.
    M, D = 4, 2048
    A0, _ = inputs.make_problem(M, D, D, seed=12)
    Ws = [inputs.make_problem(M, D, D, seed=40 + i)[1] for i in range(6)]
    Wd = [w.to(DEV) for w in Ws]
    Cs = [A0.to(DEV)] + [torch.empty((M, D), dtype=torch.bfloat16, device=DEV) for _ in Ws]
    for i, w in enumerate(Wd):
        st = lowm.lowm_gemm_bf16_ex(Cs[i], w, Cs[i + 1], M, D, D, 2, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT, None)
        assert st == lowm.LOWM_OK
    sync_ok()
    for i, w in enumerate(Wd):
        ref = torch.empty((M, D), dtype=torch.bfloat16, device=DEV)
        assert lowm.lowm_gemm_bf16(Cs[i], w, ref, M, D, D, 2, None) == lowm.LOWM_OK
        sync_ok()
        assert torch.equal(ref.view(torch.int16), Cs[i + 1].view(torch.int16)), "link %d" % i


@pytest.mark.parametrize("M1,N1,K1,N2,K2", [(128, 4096, 2048, 128, 4096), (128, 6144, 1024, 768, 1024),
                                              (64, 6144, 4096, 3072, 128)])
def test_w_written_by_the_previous_gemm_without_the_promise(M1, N1, K1, N2, K2):
    # Without the W promise a CTA requests the first stages of W into L2
    # before the dependency wait.  Here W of the second GEMM is the first
    # GEMM's output, launched back to back with no synchronization between
    # them, so those requests can run while the first GEMM still writes W:
    # the second GEMM must read W as the first one left it (a separate launch
    # after a synchronization gives the same bits, and the oracle agrees).
    st, t = lowm.lowm_gemm_query_tactic(4, N2, K2, 0)
    assert st == lowm.LOWM_OK and t["l2_before_wait_stages"] >= 1 and t["w_prefetch_stages"] == 0
    A1, W1 = inputs.make_problem(M1, N1, K1, seed=71)
    A2, _ = inputs.make_problem(4, N2, K2, seed=72)
    A1d, W1d, A2d = A1.to(DEV), W1.to(DEV), A2.to(DEV)
    for rep in range(3):
        C1 = torch.full((M1, N1), float("nan"), dtype=torch.bfloat16, device=DEV)
        C2 = torch.empty((4, N2), dtype=torch.bfloat16, device=DEV)
        assert lowm.lowm_gemm_bf16(A1d, W1d, C1, M1, N1, K1, 0, None) == lowm.LOWM_OK
        assert lowm.lowm_gemm_bf16(A2d, C1.view(N2, K2), C2, 4, N2, K2, 0, None) == lowm.LOWM_OK
        sync_ok()
        ref = torch.empty((4, N2), dtype=torch.bfloat16, device=DEV)
        assert lowm.lowm_gemm_bf16(A2d, C1.view(N2, K2), ref, 4, N2, K2, 0, None) == lowm.LOWM_OK
        sync_ok()
        assert torch.equal(ref.view(torch.int16), C2.view(torch.int16)), "repeat %d" % rep
    C = check(A2, C1.view(N2, K2).cpu(), 0)                # the synchronized launch meets the parity bar
    assert np.array_equal(C, inputs.bits(C2.cpu()))


@pytest.mark.parametrize("M,N,K,split_k", [(4, 6144, 4096, 2), (4, 49152, 4096, 2), (64, 192, 1024, 8),
                                           (3, 64, 64, 1)])
def test_w_before_pdl_wait_flag_gives_the_same_bits(M, N, K, split_k):
    A, W = inputs.make_problem(M, N, K, seed=13)
    Ad, Wd = A.to(DEV), W.to(DEV)
    c0 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    c1 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16(Ad, Wd, c0, M, N, K, split_k, None) == lowm.LOWM_OK
    assert lowm.lowm_gemm_bf16_ex(Ad, Wd, c1, M, N, K, split_k, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT, None) \
        == lowm.LOWM_OK
    sync_ok()
    assert torch.equal(c0.view(torch.int16), c1.view(torch.int16))


@pytest.mark.parametrize("prefetch", ["0", "1", "2", "3"])
def test_every_prefetch_depth_gives_the_same_bits(prefetch, monkeypatch):
    # The number of W stages requested before the dependency wait changes only timing.
    M, N, K, split_k = 4, 6144, 4096, 2
    A, W = inputs.make_problem(M, N, K, seed=21)
    Ad, Wd = A.to(DEV), W.to(DEV)
    c0 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    c1 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16(Ad, Wd, c0, M, N, K, split_k, None) == lowm.LOWM_OK
    monkeypatch.setenv("LOWM_W_PREFETCH", prefetch)
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, split_k, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    assert t["w_prefetch_stages"] == min(int(prefetch), t["stages"])
    for _ in range(3):
        assert lowm.lowm_gemm_bf16_ex(Ad, Wd, c1, M, N, K, split_k, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT, None) \
            == lowm.LOWM_OK
    sync_ok()
    assert torch.equal(c0.view(torch.int16), c1.view(torch.int16))


@pytest.mark.parametrize("split_k", [1, 2, 4])
@pytest.mark.parametrize("tile", ["64", "128"])
def test_identity_weight_covers_every_k_step(split_k, tile, monkeypatch):
    # W[n, k] = 1 iff k == n with N = K: output column n is input column n, so
    # every 16-wide K step of every block and stage (both MMA issuers' shares)
    # must land in the sum exactly once.
    monkeypatch.setenv("LOWM_TILE_N", tile)
    M, N, K = 16, 512, 512
    A = (torch.arange(M * K, dtype=torch.float32).reshape(M, K) % 241 - 120).to(torch.bfloat16)
    W = torch.zeros((N, K), dtype=torch.bfloat16)
    W[torch.arange(N), torch.arange(N)] = 1.0
    C, F = run_gpu(A, W, split_k)
    assert np.array_equal(C, inputs.bits(A)), "an output column does not hold its own input column"
    assert np.array_equal(F, A.to(torch.float64).numpy())


# ---------------------------------------------------------------- persistent schedule
PERSISTENT = [
    # M, N, K, split_k, max clusters: several tiles per cluster, uneven tile counts, ring wrap across tiles
    (4, 13 * 64, 1024, 2, 4), (1, 7 * 64, 512, 1, 3), (8, 9 * 64, 2048, 4, 2), (5, 10 * 64, 1024, 8, 3),
    (16, 6 * 64, 4096, 2, 2), (32, 5 * 64, 1024, 1, 2), (64, 6 * 64, 2048, 2, 3), (3, 2 * 64, 256, 2, 1),
]


@pytest.mark.parametrize("M,N,K,split_k,cap", PERSISTENT)
def test_persistent_schedule_random(M, N, K, split_k, cap, monkeypatch):
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", str(cap))
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK and t["persistent"] == 1 and t["num_clusters"] <= cap
    A, W = inputs.make_problem(M, N, K, seed=300 + M + N + K)
    check(A, W, split_k)


@pytest.mark.parametrize("M,N,K,split_k,cap", [(16, 12 * 64, 4096, 4, 5), (4, 11 * 64, 2048, 2, 3)])
def test_persistent_schedule_integer_exact(M, N, K, split_k, cap, monkeypatch):
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", str(cap))
    A, W = inputs.make_problem(M, N, K, seed=8, kind="int")
    check(A, W, split_k, exact=True)


def test_persistent_and_one_tile_schedules_both_meet_the_bar(monkeypatch):
    # The one-tile kernel sums two accumulators (two MMA issuers) and the
    # persistent kernel one, so their fp32 sums may differ in the last bits;
    # each must meet the parity bar and be launch-to-launch deterministic.
    M, N, K, sk = 4, 6144, 4096, 2
    A, W = inputs.make_problem(M, N, K, seed=21)
    monkeypatch.setenv("LOWM_PERSISTENT", "0")
    C0 = check(A, W, sk)
    assert np.array_equal(C0, run_gpu(A, W, sk, want_f32=False)[0])
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", "40")
    C1 = check(A, W, sk)
    assert np.array_equal(C1, run_gpu(A, W, sk, want_f32=False)[0])


# ---------------------------------------------------------------- K blocks per stage
@pytest.mark.parametrize("kbs", [1, 2, 4, 8])
@pytest.mark.parametrize("M,N,K,split_k", [(4, 640, 2048, 2), (8, 192, 4096, 1), (3, 128, 4096, 8)])
def test_every_kb_per_stage_random(kbs, M, N, K, split_k, monkeypatch):
    monkeypatch.setenv("LOWM_KB_PER_STAGE", str(kbs))
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK and t["kb_per_stage"] == kbs
    A, W = inputs.make_problem(M, N, K, seed=500 + kbs + M)
    check(A, W, split_k)


@pytest.mark.parametrize("M,N,K,split_k", [(4, 256, 64 * 3, 1), (5, 128, 64 * 5, 1), (16, 192, 64 * 6, 1),
                                           (64, 128, 64 * 12, 2), (33, 64, 64 * 14, 2)])
def test_block_counts_not_divisible_by_four(M, N, K, split_k):
    A, W = inputs.make_problem(M, N, K, seed=600 + K)
    check(A, W, split_k)


@pytest.mark.parametrize("kbs", [1, 4])
def test_kb_per_stage_integer_exact(kbs, monkeypatch):
    monkeypatch.setenv("LOWM_KB_PER_STAGE", str(kbs))
    A, W = inputs.make_problem(16, 256, 4096, seed=9, kind="int")
    check(A, W, 2, exact=True)


@pytest.mark.parametrize("kbs", [1, 4])
def test_persistent_with_kb_per_stage(kbs, monkeypatch):
    monkeypatch.setenv("LOWM_KB_PER_STAGE", str(kbs))
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", "5")
    A, W = inputs.make_problem(4, 17 * 64, 2048, seed=10)
    check(A, W, 2)


# ---------------------------------------------------------------- 128-column tiles (MMA M = 128)
def test_identity_weight_maps_every_column_tile128(monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", "128")
    M, N, K = 8, 128, 256
    A = (torch.arange(M * K, dtype=torch.float32).reshape(M, K) % 251 + 1).to(torch.bfloat16)
    W = torch.zeros((N, K), dtype=torch.bfloat16)
    W[torch.arange(N), torch.arange(N)] = 1.0
    for split_k in (1, 2):
        st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
        assert st == lowm.LOWM_OK and t["tile_n"] == 128
        C, _ = run_gpu(A, W, split_k, want_f32=False)
        want = inputs.bits(A)[:, :N]
        if not np.array_equal(C, want):
            vals = {int(v): i for i, v in enumerate(want[0])}
            got_cols = [vals.get(int(v), -1) for v in C[0]]
            raise AssertionError("split_k %d: output column n holds input column %s" % (split_k, got_cols))


TILE128 = [
    (1, 128, 256, 1), (4, 384, 1024, 2), (13, 256, 2048, 4), (16, 128, 4096, 8), (17, 256, 512, 2),
    (32, 384, 1024, 1), (33, 128, 768, 2), (64, 256, 2048, 4), (4, 6144, 4096, 2), (8, 1280, 64 * 12, 4),
]


@pytest.mark.parametrize("M,N,K,split_k", TILE128)
def test_tile128_random(M, N, K, split_k, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", "128")
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK
    A, W = inputs.make_problem(M, N, K, seed=700 + M + N + K)
    check(A, W, split_k)


@pytest.mark.parametrize("M,N,K,split_k", [(16, 6144, 32768, 4), (4, 256, 4096, 2), (64, 128, 1024, 1)])
def test_tile128_integer_exact(M, N, K, split_k, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", "128")
    A, W = inputs.make_problem(M, N, K, seed=11, kind="int")
    check(A, W, split_k, exact=True)


def test_tile128_persistent(monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", "128")
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", "3")
    st, t = lowm.lowm_gemm_query_tactic(4, 11 * 128, 2048, 2)
    assert st == lowm.LOWM_OK and t["tile_n"] == 128 and t["persistent"] == 1
    A, W = inputs.make_problem(4, 11 * 128, 2048, seed=12)
    check(A, W, 2)


def test_tile64_and_tile128_agree_within_tolerance(monkeypatch):
    A, W = inputs.make_problem(4, 1024, 4096, seed=13)
    monkeypatch.setenv("LOWM_TILE_N", "64")
    C64 = check(A, W, 2)
    monkeypatch.setenv("LOWM_TILE_N", "128")
    C128 = check(A, W, 2)
    assert C64.shape == C128.shape                      # both met the parity bar inside check()


# ---------------------------------------------------------------- N not a multiple of the tile width
NTAIL = [
    # M, N, K, split_k: a partial last tile, with N % 8 == 0 (16-byte stores) and N % 8 != 0 (element stores)
    (4, 1, 256, 1), (3, 8, 512, 2), (4, 72, 1024, 2), (5, 100, 512, 1), (8, 200, 2048, 4),
    (16, 6152, 1024, 2), (16, 6150, 1024, 2), (33, 130, 512, 1), (64, 136, 1024, 2), (1, 4095, 256, 1),
]


@pytest.mark.parametrize("M,N,K,split_k", NTAIL)
def test_n_tail_random(M, N, K, split_k):
    A, W = inputs.make_problem(M, N, K, seed=500 + M + N)
    check(A, W, split_k)


@pytest.mark.parametrize("N", [72, 100, 6150])
def test_n_tail_writes_nothing_past_n(N):
    # C is the head of a larger buffer: the elements after C[M-1, N-1] must keep their sentinel.
    M, K = 5, 1024
    A, W = inputs.make_problem(M, N, K, seed=31)
    flat = torch.full((M * N + 512,), 7.0, dtype=torch.bfloat16, device=DEV)
    C = flat[:M * N].view(M, N)
    F = torch.empty((M, N), dtype=torch.float32, device=DEV)
    assert lowm.lowm_gemm_bf16_debug(A.to(DEV), W.to(DEV), C, M, N, K, 2, None, c_f32=F) == lowm.LOWM_OK
    sync_ok()
    assert torch.all(flat[M * N:] == 7.0)
    Cref, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert_parity(inputs.bits(C.cpu()), F.cpu().numpy().astype(np.float64), Cref, S, A, W)


@pytest.mark.parametrize("tile", ["64", "128"])
def test_n_tail_integer_exact(tile, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", tile)
    M, N, K = 16, 6150, 4096
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, 2)
    assert st == lowm.LOWM_OK and t["tile_n"] == int(tile) and t["tiles"] == -(-N // int(tile))
    A, W = inputs.make_problem(M, N, K, seed=9, kind="int")
    C = check(A, W, 2, exact=True)
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(C, np.broadcast_to(inputs.bits(col[None, :]), C.shape))


@pytest.mark.parametrize("tile", ["64", "128"])
def test_n_tail_persistent(tile, monkeypatch):
    monkeypatch.setenv("LOWM_PERSISTENT", "1")
    monkeypatch.setenv("LOWM_MAX_CLUSTERS", "3")
    monkeypatch.setenv("LOWM_TILE_N", tile)
    M, N, K = 16, 10 * 128 + 40, 2048
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, 2)
    assert st == lowm.LOWM_OK and t["persistent"] == 1 and t["tiles_per_cluster"] >= 2
    A, W = inputs.make_problem(M, N, K, seed=14)
    check(A, W, 2)


def test_largest_k_and_split():
    # K = 65536 (the oracle's exact accumulator bound) over a cluster of 8.
    A, W = inputs.make_problem(4, 256, 65536, seed=15)
    check(A, W, 8)


# ---------------------------------------------------------------- 65 <= M <= 128 (m_pad 96 / 128, chunked epilogue)
MBIG = [
    # M, N, K, split_k: every split with an m_pad 96 or 128 instance, ragged M and N, ring wrap-around
    (65, 192, 1024, 1), (80, 256, 2048, 2), (96, 640, 1024, 4), (127, 130, 512, 2), (128, 128, 4096, 1),
    (100, 4095, 256, 1), (128, 6144, 4096, 0), (96, 6144, 4096, 0), (72, 2000, 1024, 3), (90, 1024, 2048, 2),
    (97, 640, 1024, 3),
]


# ---------------------------------------------------------------- 33 <= M <= 48 (m_pad 48)
@pytest.mark.parametrize("M,N,K,split_k", [(33, 192, 1024, 1), (40, 640, 2048, 2), (48, 6144, 4096, 0),
                                           (41, 2000, 1024, 3), (48, 256, 2048, 4), (36, 192, 1024, 8),
                                           (44, 70, 512, 2)])
def test_m_pad_48_random(M, N, K, split_k):
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK and t["m_pad"] == 48
    A, W = inputs.make_problem(M, N, K, seed=760 + M + N)
    check(A, W, split_k)


@pytest.mark.parametrize("tile,split_k", [("64", 1), ("64", 2), ("64", 8), ("128", 2), ("128", 4)])
def test_m_pad_48_integer_exact(tile, split_k, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", tile)
    M, N, K = 48, 1024, 4096
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK and t["tile_n"] == int(tile) and t["m_pad"] == 48
    A, W = inputs.make_problem(M, N, K, seed=18, kind="int")
    C = check(A, W, split_k, exact=True)
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(C, np.broadcast_to(inputs.bits(col[None, :]), C.shape))


@pytest.mark.parametrize("M,N,K,split_k", MBIG)
def test_m_up_to_128_random(M, N, K, split_k):
    A, W = inputs.make_problem(M, N, K, seed=700 + M + N)
    check(A, W, split_k)


@pytest.mark.parametrize("M", [96, 128])
@pytest.mark.parametrize("tile,split_k", [("64", 1), ("64", 2), ("64", 4), ("128", 1), ("128", 2)])
def test_m_up_to_128_integer_exact(M, tile, split_k, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", tile)
    N, K = 1024, 4096
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK and t["tile_n"] == int(tile) and t["m_pad"] == M
    A, W = inputs.make_problem(M, N, K, seed=17, kind="int")
    C = check(A, W, split_k, exact=True)
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(C, np.broadcast_to(inputs.bits(col[None, :]), C.shape))


@pytest.mark.parametrize("M", [96, 128])
@pytest.mark.parametrize("tile,split_k", [("64", 1), ("64", 4), ("128", 2), ("128", 3)])
def test_identity_weight_m128_maps_every_row_and_column(M, tile, split_k, monkeypatch):
    # Distinct rows of A (integers) and W = I: C[m, n] = A[m, n] exactly, which
    # pins the m_pad 96 / 128 column chunks of the accumulators and the mailbox.
    monkeypatch.setenv("LOWM_TILE_N", tile)
    N, K = 512, 512
    A = ((torch.arange(M * K, dtype=torch.float32).reshape(M, K) * 7) % 251 - 125).to(torch.bfloat16)
    W = torch.zeros((N, K), dtype=torch.bfloat16)
    W[torch.arange(N), torch.arange(N)] = 1.0
    C, F = run_gpu(A, W, split_k)
    assert np.array_equal(C, inputs.bits(A)[:, :N])
    assert np.array_equal(F, A.to(torch.float64).numpy()[:, :N])


@pytest.mark.parametrize("M", [96, 128])
def test_m128_twenty_launches_are_bitwise_identical(M):
    N, K, split_k = 6144, 4096, 2
    A, W = inputs.make_problem(M, N, K, seed=33)
    Ad, Wd = A.to(DEV), W.to(DEV)
    outs = torch.empty((20, M, N), dtype=torch.bfloat16, device=DEV)
    for i in range(20):
        assert lowm.lowm_gemm_bf16(Ad, Wd, outs[i], M, N, K, split_k, None) == lowm.LOWM_OK
    sync_ok()
    o = outs.view(torch.int16)
    assert bool((o == o[0:1]).all())
    C = check(A, W, split_k)                      # the same launch configuration against the oracle
    assert np.array_equal(C, inputs.bits(outs[0].cpu()))


# ---------------------------------------------------------------- large grids and the Python convenience wrapper
@pytest.mark.parametrize("M,N,K,split_k", [(4, 1 << 20, 64, 1), (3, (1 << 19) + 40, 128, 2), (128, 1 << 17, 64, 1)])
def test_large_grids(M, N, K, split_k):
    # Tens of thousands of CTAs (16384 clusters at N 2^20), a ragged last tile
    # and the largest m_pad, each against the oracle element by element.
    A, W = inputs.make_problem(M, N, K, seed=44)
    check(A, W, split_k)


def test_python_gemm_wrapper_allocates_and_raises():
    M, N, K = 5, 384, 1024
    A, W = inputs.make_problem(M, N, K, seed=45)
    C = lowm.gemm(A.to(DEV), W.to(DEV), split_k=2)
    sync_ok()
    assert C.shape == (M, N) and C.dtype == torch.bfloat16
    Cref, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    F = torch.empty((M, N), dtype=torch.float32, device=DEV)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.lowm_gemm_bf16_debug(A.to(DEV), W.to(DEV), Cd, M, N, K, 2, None, c_f32=F) == lowm.LOWM_OK
    sync_ok()
    assert torch.equal(C.view(torch.int16), Cd.view(torch.int16))       # the wrapper runs the same kernel
    assert_parity(inputs.bits(C.cpu()), F.cpu().numpy().astype(np.float64), Cref, S, A, W)
    C2 = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    assert lowm.gemm(A.to(DEV), W.to(DEV), C2, split_k=2) is C2
    sync_ok()
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
    C3 = lowm.gemm(A.to(DEV), W.to(DEV), split_k=2, flags=lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)   # the W promise
    sync_ok()
    assert torch.equal(C.view(torch.int16), C3.view(torch.int16))
    with pytest.raises(lowm.LowmError) as e:
        lowm.gemm(A.to(DEV), W.to(DEV), split_k=2, flags=4)                 # unknown flag bit
    assert e.value.status == lowm.LOWM_ERR_INVALID_ARGUMENT
    with pytest.raises(lowm.LowmError) as e:
        lowm.gemm(A.to(DEV)[:, :96].contiguous(), W.to(DEV)[:, :96].contiguous(), split_k=1)   # K = 96: not a multiple of 64
    assert e.value.status == lowm.LOWM_ERR_UNSUPPORTED_SHAPE


# ---------------------------------------------------------------- seeded fuzz over shapes and tactic overrides
def _fuzz_cases(n=60, seed=20261202):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        M = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64, 65, 100, 127, 128]))
        sk = int(rng.choice([1, 2, 4, 8]))
        K = 64 * sk * int(rng.integers(1, 9))
        N = int(rng.choice([int(rng.integers(1, 700)), 64 * int(rng.integers(1, 12))]))
        env = {"LOWM_TILE_N": str(int(rng.choice([0, 64, 128]))),
               "LOWM_KB_PER_STAGE": str(int(rng.choice([0, 1, 2, 4, 8]))),
               "LOWM_STAGES": str(int(rng.choice([0, 2, 3, 4, 6]))),
               "LOWM_W_PREFETCH": str(int(rng.choice([-1, 0, 1, 2])))}
        flags = int(rng.integers(0, 2))
        cases.append((M, N, K, sk, env, flags))
    return cases


@pytest.mark.parametrize("case", range(60))
def test_fuzz_shapes_and_tactics(case, monkeypatch):
    M, N, K, sk, env, flags = _fuzz_cases()[case]
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    if st == lowm.LOWM_ERR_UNSUPPORTED_SHAPE:
        # only shapes whose mailbox or forced ring cannot fit may be refused
        assert (M > 64 and sk == 8) or env["LOWM_STAGES"] != "0" or env["LOWM_KB_PER_STAGE"] != "0"
        pytest.skip("refused by the host before any launch: %s" % lowm.status_string(st))
    assert st == lowm.LOWM_OK
    A, W = inputs.make_problem(M, N, K, seed=900 + case)
    Ad, Wd = A.to(DEV), W.to(DEV)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    F = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    assert lowm.lowm_gemm_bf16_debug(Ad, Wd, C, M, N, K, sk, None, c_f32=F, flags=flags) == lowm.LOWM_OK
    sync_ok()
    Cref, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert_parity(inputs.bits(C.cpu()), F.cpu().numpy().astype(np.float64), Cref, S, A, W)


# ---------------------------------------------------------------- split_k 3 (uneven K shares) and the ring-aliased mailbox
SPLIT3 = [
    # M, N, K, tile: stage counts that 3 does not divide (the first ranks take one stage fewer), every m_pad
    (1, 192, 64 * 4, "64"), (4, 640, 64 * 7, "64"), (8, 256, 64 * 64, "64"), (13, 384, 64 * 10, "128"),
    (16, 6144, 4096, "128"), (32, 320, 64 * 11, "64"), (48, 256, 64 * 5, "128"), (64, 6144, 4096, "128"),
    (64, 192, 64 * 3, "64"), (100, 130, 64 * 8, "64"), (128, 6144, 4096, "128"), (128, 6144, 4096, "64"),
]


@pytest.mark.parametrize("M,N,K,tile", SPLIT3)
def test_split3_random(M, N, K, tile, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", tile)
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, 3)
    assert st == lowm.LOWM_OK and t["split_k"] == 3 and t["mbox_in_ring"] == 1
    A, W = inputs.make_problem(M, N, K, seed=1100 + M + N + K)
    check(A, W, 3)


@pytest.mark.parametrize("M,tile", [(4, "64"), (16, "128"), (64, "128"), (128, "64"), (128, "128")])
def test_split3_integer_exact(M, tile, monkeypatch):
    monkeypatch.setenv("LOWM_TILE_N", tile)
    N, K = 1024, 64 * 50                               # 50 blocks: shares of 16/17 blocks or whole uneven stages
    A, W = inputs.make_problem(M, N, K, seed=19, kind="int")
    C = check(A, W, 3, exact=True)
    col = W.to(torch.int64).sum(dim=1).to(torch.float32).to(torch.bfloat16)
    assert np.array_equal(C, np.broadcast_to(inputs.bits(col[None, :]), C.shape))


@pytest.mark.parametrize("kbs", ["1", "2", "4"])
@pytest.mark.parametrize("tile", ["64", "128"])
def test_split3_identity_weight_covers_every_k_step(kbs, tile, monkeypatch):
    # W = I with N = K: every 16-wide K step of every rank's (uneven) share
    # must land in the sum exactly once, whatever the stage size.
    monkeypatch.setenv("LOWM_TILE_N", tile)
    monkeypatch.setenv("LOWM_KB_PER_STAGE", kbs)
    M, N, K = 16, 64 * 20, 64 * 20                     # 20 blocks: 5, 10 or 20 stages, none divisible by 3
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, 3)
    assert st == lowm.LOWM_OK and t["kb_per_stage"] == int(kbs)
    A = (torch.arange(M * K, dtype=torch.float32).reshape(M, K) % 241 - 120).to(torch.bfloat16)
    W = torch.zeros((N, K), dtype=torch.bfloat16)
    W[torch.arange(N), torch.arange(N)] = 1.0
    C, F = run_gpu(A, W, 3)
    assert np.array_equal(C, inputs.bits(A)), "an output column does not hold its own input column"
    assert np.array_equal(F, A.to(torch.float64).numpy())


@pytest.mark.parametrize("M,N,K,split_k", [(4, 640, 64 * 6, 2), (64, 256, 2048, 2), (128, 384, 2048, 4),
                                           (16, 6144, 4096, 2), (64, 1024, 64 * 3, 2)])
def test_mailbox_in_ring_for_even_splits(M, N, K, split_k, monkeypatch):
    # The aliased mailbox with split_k 2 and 4 (and an uneven split 2 of 3 blocks).
    monkeypatch.setenv("LOWM_MBOX_IN_RING", "1")
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, split_k)
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == 1
    A, W = inputs.make_problem(M, N, K, seed=1200 + M + K)
    check(A, W, split_k)


def test_mailbox_next_to_ring_for_split3(monkeypatch):
    monkeypatch.setenv("LOWM_MBOX_IN_RING", "0")
    st, t = lowm.lowm_gemm_query_tactic(8, 640, 64 * 9, 3)
    assert st == lowm.LOWM_OK and t["mbox_in_ring"] == 0
    A, W = inputs.make_problem(8, 640, 64 * 9, seed=1300)
    check(A, W, 3)


@pytest.mark.parametrize("M,tile", [(4, "64"), (64, "128"), (128, "128")])
def test_split3_dropped_mailbox_times_out(M, tile, monkeypatch):
    # The peers skip their publication into the aliased mailbox: the owner's
    # bounded waits run out, report the mailbox bit, and the context survives.
    monkeypatch.setenv("LOWM_TILE_N", tile)
    N, K = 256, 64 * 12
    A, W = inputs.make_problem(M, N, K, seed=6)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    st = lowm.lowm_gemm_bf16_debug(A.to(DEV), W.to(DEV), C, M, N, K, 3, None, drop_mailbox=1,
                                   reduce_timeout_ns=20_000_000)
    assert st == lowm.LOWM_OK
    st, detail = lowm.lowm_gemm_sync_status()
    assert st == lowm.LOWM_ERR_TIMEOUT and detail == (1 << 8), (st, hex(detail))
    check(A, W, 3)


@pytest.mark.parametrize("M,N,K", [(64, 6144, 4096), (128, 6144, 4096)])
def test_split3_twenty_launches_are_bitwise_identical(M, N, K):
    A, W = inputs.make_problem(M, N, K, seed=34)
    Ad, Wd = A.to(DEV), W.to(DEV)
    outs = torch.empty((20, M, N), dtype=torch.bfloat16, device=DEV)
    for i in range(20):
        assert lowm.lowm_gemm_bf16(Ad, Wd, outs[i], M, N, K, 3, None) == lowm.LOWM_OK
    sync_ok()
    o = outs.view(torch.int16)
    assert bool((o == o[0:1]).all())


# ---------------------------------------------------------------- seeded fuzz over uneven K shares, the mailbox placement and the L2 prefetch
def _fuzz_cases_uneven(n=40, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        M = int(rng.choice([1, 3, 4, 8, 9, 16, 17, 32, 40, 64, 65, 96, 128]))
        sk = int(rng.choice([2, 3, 4, 8]))
        K = 64 * int(rng.integers(sk, 9 * sk + 1))           # any block count with a non-empty share per rank
        N = int(rng.choice([int(rng.integers(1, 600)), 128 * int(rng.integers(1, 8))]))
        env = {"LOWM_TILE_N": str(int(rng.choice([0, 64, 128]))),
               "LOWM_KB_PER_STAGE": str(int(rng.choice([0, 1, 2, 4]))),
               "LOWM_MBOX_IN_RING": str(int(rng.choice([-1, 0, 1]))),
               "LOWM_L2_PREFETCH": str(int(rng.choice([-1, 0, 1, 2, 3])))}
        cases.append((M, N, K, sk, env, int(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("case", range(40))
def test_fuzz_uneven_splits_mailbox_and_prefetch(case, monkeypatch):
    M, N, K, sk, env, flags = _fuzz_cases_uneven()[case]
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    st, t = lowm.lowm_gemm_query_tactic(M, N, K, sk)
    if st == lowm.LOWM_ERR_UNSUPPORTED_SHAPE:
        # only a mailbox that cannot fit next to the ring may be refused
        assert M > 64 or env["LOWM_MBOX_IN_RING"] == "0"
        pytest.skip("refused by the host before any launch: %s" % lowm.status_string(st))
    assert st == lowm.LOWM_OK
    A, W = inputs.make_problem(M, N, K, seed=1500 + case)
    Ad, Wd = A.to(DEV), W.to(DEV)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    F = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    assert lowm.lowm_gemm_bf16_debug(Ad, Wd, C, M, N, K, sk, None, c_f32=F, flags=flags) == lowm.LOWM_OK
    sync_ok()
    Cref, S = oracle.gemm_bf16_f64(inputs.bits(A), inputs.bits(W))
    assert_parity(inputs.bits(C.cpu()), F.cpu().numpy().astype(np.float64), Cref, S, A, W,
                  label="fuzz-uneven %d" % case)


# ---------------------------------------------------------------- the timed launches: with the W-before-PDL promise
@pytest.mark.parametrize("M,N,K,split_k,kind", [
    (4, 6144, 4096, 2, "randn"), (4, 2304, 12288, 4, "randn"), (4, 49152, 4096, 2, "randn"),
    (16, 6144, 32768, 4, "int"), (1, 6144, 4096, 0, "randn"), (16, 6144, 4096, 0, "randn"),
    (32, 6144, 4096, 0, "randn"), (64, 6144, 4096, 0, "randn"), (128, 6144, 4096, 0, "randn")])
def test_workloads_with_the_w_promise(M, N, K, split_k, kind):
    # The tactic the benchmark times (lowm_gemm_bf16_ex with
    # LOWM_FLAG_W_BEFORE_PDL_WAIT: deeper rings, the mailbox in the ring)
    # against the oracle, and bitwise equal to the launch without the flag.
    st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, split_k, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    assert st == lowm.LOWM_OK
    A, W = inputs.make_problem(M, N, K, seed=1800 + M, kind=kind)
    C1 = check(A, W, split_k, exact=(kind == "int"), flags=lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    C0, _ = run_gpu(A, W, split_k, want_f32=False)
    assert np.array_equal(C0, C1)


@pytest.mark.parametrize("M,N,K,tile,split_k", [
    (4, 4096, 4096, 128, 2), (4, 2048, 8192, 128, 4), (4, 1024, 16384, 64, 4), (4, 8192, 4096, 128, 2),
    (16, 6144, 16384, 128, 4), (64, 12288, 8192, 128, 2), (4, 1536, 8192, 64, 4)])
def test_auto_tactics_of_the_tile_sweep(M, N, K, tile, split_k):
    # The tactics the 128-column rule and the auto split pick across shapes
    # (64 to two-per-SM CTAs, 512 KiB of W per CTA, long K), with and without
    # the W promise, against the oracle.
    for flags in (0, lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT):
        st, t = lowm.lowm_gemm_query_tactic_ex(M, N, K, 0, flags)
        assert st == lowm.LOWM_OK and (t["tile_n"], t["split_k"]) == (tile, split_k)
    A, W = inputs.make_problem(M, N, K, seed=1900 + M + N // 64)
    C1 = check(A, W, 0, flags=lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    C0, _ = run_gpu(A, W, 0, want_f32=False)
    assert np.array_equal(C0, C1)


@pytest.mark.parametrize("M,N,K,split_k", [(4, 6144, 4096, 2), (64, 6144, 4096, 0), (4, 2304, 12288, 4),
                                           (96, 1024, 2048, 2), (3, 200, 640, 3)])
def test_gemms_sharing_a_with_both_promises(M, N, K, split_k):
    # Projections of one input: A is shared and never written, each GEMM has
    # its own W, launched back to back with both promises (A and W loaded
    # without waiting for the preceding GEMM; only C waits).  Each output
    # equals a launch without flags on the same operands, and the first one
    # meets the parity bar.
    both = lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT | lowm.LOWM_FLAG_A_BEFORE_PDL_WAIT
    A, _ = inputs.make_problem(M, N, K, seed=91)
    Ws = [inputs.make_problem(M, N, K, seed=92 + i)[1] for i in range(4)]
    Ad = A.to(DEV)
    Wd = [w.to(DEV) for w in Ws]
    Cs = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in Ws]
    for w, c in zip(Wd, Cs):
        assert lowm.lowm_gemm_bf16_ex(Ad, w, c, M, N, K, split_k, both, None) == lowm.LOWM_OK
    sync_ok()
    for w, c in zip(Wd, Cs):
        ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        assert lowm.lowm_gemm_bf16(Ad, w, ref, M, N, K, split_k, None) == lowm.LOWM_OK
        sync_ok()
        assert torch.equal(ref.view(torch.int16), c.view(torch.int16))
    C = check(A, Ws[0], split_k, flags=both)
    assert np.array_equal(C, inputs.bits(Cs[0].cpu()))


def test_pdl_chain_with_the_deep_ring_and_w_promise():
    # C of each GEMM is the next GEMM's A (K = N = 6144), launched back to back
    # with the W promise: the 128-column tactic with the 4 x 3 ring and the
    # mailbox in the ring requests W before the dependency wait, and must
    # still read A only after it.  Each link must equal a separate launch on
    # the same input, which itself meets the parity bar.
    M, D = 4, 6144
    flags = lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT
    st, t = lowm.lowm_gemm_query_tactic_ex(M, D, D, 2, flags)
    assert st == lowm.LOWM_OK and t["tile_n"] == 128 and t["mbox_in_ring"] == 1 and t["w_prefetch_stages"] >= 2
    A0, _ = inputs.make_problem(M, D, D, seed=51)
    Ws = [inputs.make_problem(M, D, D, seed=60 + i)[1] for i in range(4)]
    Wd = [w.to(DEV) for w in Ws]
    Cs = [A0.to(DEV)] + [torch.empty((M, D), dtype=torch.bfloat16, device=DEV) for _ in Ws]
    for i, w in enumerate(Wd):
        assert lowm.lowm_gemm_bf16_ex(Cs[i], w, Cs[i + 1], M, D, D, 2, flags, None) == lowm.LOWM_OK
    sync_ok()
    for i, w in enumerate(Ws):
        a = Cs[i].cpu()
        alone = check(a, w, 2, flags=flags)                # a separate launch on this link's input, vs the oracle
        assert np.array_equal(inputs.bits(Cs[i + 1].cpu()), alone), "link %d" % i
