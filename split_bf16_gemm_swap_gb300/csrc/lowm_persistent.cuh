// Persistent form of the low-M split-K GEMM for shapes with more 64-column
// tiles than resident clusters (e.g. N = 49152: 768 tiles).
//
// The method is the same as lowm_splitk_kernel (same warp roles, swap-AB
// tcgen05.mma, cluster mailbox with a relaxed cluster-scope wait plus an
// acquire fence restricted to shared::cluster, the fixed two-phase TMEM
// release from "Fix two synchronization gaps in the MiniMax M3 low-M split-K
// GEMM", Description items 1 and 2).  What changes is the schedule:
//   - cluster c owns tiles c, c + G, c + 2G, ... (G = clusters launched, chosen
//     on the host so every cluster gets the same number of tiles);
//   - the TMA ring streams the cluster's whole K range tile after tile without
//     draining, so there is one prologue and one pipeline fill per CTA;
//   - the TMEM accumulator, the owner's mailbox and the output staging are
//     double-buffered by tile parity, so tile j's epilogue (load, exchange,
//     store) overlaps tile j+1's MMAs.
// Extra barriers for the double buffers:
//   acc_full[b]   count 1    tcgen05.commit after a tile's last MMA
//   acc_empty[b]  count 128  epilogue threads, after tcgen05.wait::ld of that buffer
//   reduce[b]     count 1    owner: armed with expect_tx; peers' st.async complete_tx
//   mbox_free[b]  count 1    peers: the owner's remote arrive once it has read set b
// A buffer's u-th use waits for parity (u & 1) on its "full" barriers and for
// parity (u & 1) ^ 1 on its "empty"/"free" barriers (a fresh barrier reports
// the parity-1 phase as complete, so first uses pass at once).
#pragma once

#include "lowm_kernel.cuh"

namespace lowm {

template <int TILE_N, int M_PAD, int SPLIT_K>
__global__ void __launch_bounds__(kThreadsPersistent, 1)
    lowm_splitk_persistent_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                  const __grid_constant__ CUtensorMap tmap_w, const KernelParams p)
{
    static_assert(TILE_N == 64 || TILE_N == 128, "tile_n is the MMA M");
    static_assert(M_PAD % (TILE_N == 128 ? 16 : 8) == 0 && M_PAD >= 8 && M_PAD <= 64,
                  "m_pad is the MMA N: a multiple of 8 (M = 64) or 16 (M = 128), at most 64");
    constexpr int kTileN = TILE_N;
    static_assert(SPLIT_K == 1 || SPLIT_K == 2 || SPLIT_K == 4 || SPLIT_K == 8, "split_k");
    constexpr uint32_t kBufCols = M_PAD;                          // one tile's accumulator
    constexpr uint32_t kTmemCols = tmem_cols_for(2 * kBufCols);
    constexpr uint32_t kSlotBytes = kTileN * M_PAD * 4u;
    constexpr uint32_t kSetBytes = (SPLIT_K - 1) * kSlotBytes;    // one mailbox buffer
    constexpr uint32_t kOutBytes = M_PAD * kTileN * 2u;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int kbs = p.kb_per_stage;
    const SmemLayout L = make_smem_layout(TILE_N, M_PAD, SPLIT_K, p.stages, kbs, 2);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int stages = p.stages;
    const uint32_t w_stage_bytes = (uint32_t)kbs * w_block_bytes(TILE_N);
    const uint32_t a_stage_bytes = (uint32_t)kbs * (M_PAD * 128u);
    const uint32_t stage_tx = w_stage_bytes + a_stage_bytes;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = SPLIT_K > 1 ? ptx::cluster_ctarank() : 0u;
    const int cluster = (int)(blockIdx.x / SPLIT_K);
    const int clusters = (int)(gridDim.x / SPLIT_K);
    const int my_tiles = cluster < p.num_tiles ? (p.num_tiles - cluster + clusters - 1) / clusters : 0;
    const int kbr = p.kb_per_rank;
    const int spt = kbr / kbs;                                     // stages per tile
    const int kb0 = (int)rank * kbr;

    const uint32_t bar_full = sbase + L.bars;                      // + 8 * stage
    const uint32_t bar_empty = bar_full + 8u * stages;             // + 8 * stage
    const uint32_t bar_acc_full = bar_full + 16u * stages;         // + 8 * b
    const uint32_t bar_acc_empty = bar_acc_full + 16u;             // + 8 * b
    const uint32_t bar_tmem_alloc = bar_acc_full + 32u;            // two phases, 160 arrivals each
    const uint32_t bar_reduce = bar_acc_full + 40u;                // + 8 * b (owner)
    const uint32_t bar_mbox_free = bar_acc_full + 56u;             // + 8 * b (peers)
    const uint32_t tmem_slot = sbase + L.tmem_slot;

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(bar_full + 8u * s, 1);
            ptx::mbar_init(bar_empty + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_acc_full + 8u * b, 1);
            ptx::mbar_init(bar_acc_empty + 8u * b, kEpilogueThreads);
            ptx::mbar_init(bar_reduce + 8u * b, 1);
            ptx::mbar_init(bar_mbox_free + 8u * b, 1);
        }
        ptx::mbar_init(bar_tmem_alloc, kTmemBarArrivals);
        *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot + kTicketOffset) = 0u;
        if (SPLIT_K > 1 && rank == 0)              // arm both mailbox buffers for the first two tiles
            for (int b = 0; b < 2 && b < my_tiles; ++b)
                ptx::mbar_arrive_expect_tx(bar_reduce + 8u * b, kSetBytes);
        ptx::fence_mbarrier_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_w);
        ptx::prefetch_tensormap(&tmap_a);
    }
    if (SPLIT_K > 1) {
        ptx::cluster_arrive_release();
        ptx::cluster_wait_acquire();
    } else {
        __syncthreads();
    }
    if (p.timeline != nullptr && threadIdx.x == 0)
        p.timeline[4 * blockIdx.x] = ptx::globaltimer();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_a = ptx::policy_evict_last();
            const int total = my_tiles * spt;      // (tile, stage) pairs, tile-major
            int pre = total < stages ? total : stages;
            if (pre > (int)p.w_prefetch_stages)
                pre = (int)p.w_prefetch_stages;
            for (int i = 0; i < pre; ++i) {
                const int n0 = (cluster + (i / spt) * clusters) * kTileN;
                ptx::mbar_arrive_expect_tx(bar_full + 8u * i, stage_tx);
                ptx::tma_load_3d(sbase + L.w + (uint32_t)i * w_stage_bytes, &tmap_w, 0, n0, kb0 + (i % spt) * kbs,
                                 bar_full + 8u * i, pol_w);
            }
            ptx::griddep_wait();
            for (int i = 0; i < pre; ++i)
                ptx::tma_load_3d(sbase + L.a + (uint32_t)i * a_stage_bytes, &tmap_a, 0, 0, kb0 + (i % spt) * kbs,
                                 bar_full + 8u * i, pol_a);
            int issued = pre;
            for (int i = pre; i < total; ++i) {
                const int s = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (!wait_bounded<false>(bar_empty + 8u * s, ph ^ 1u, p.timeout_ns)) {
                    record_error(p, kErrProducerEmpty);
                    break;
                }
                const int n0 = (cluster + (i / spt) * clusters) * kTileN;
                const int kz = kb0 + (i % spt) * kbs;
                ptx::mbar_arrive_expect_tx(bar_full + 8u * s, stage_tx);
                ptx::tma_load_3d(sbase + L.w + (uint32_t)s * w_stage_bytes, &tmap_w, 0, n0, kz, bar_full + 8u * s,
                                 pol_w);
                ptx::tma_load_3d(sbase + L.a + (uint32_t)s * a_stage_bytes, &tmap_a, 0, 0, kz, bar_full + 8u * s,
                                 pol_a);
                ++issued;
            }
            ptx::griddep_launch_dependents();
            for (int j = issued > stages ? issued - stages : 0; j < issued; ++j)
                if (!wait_bounded<false>(bar_full + 8u * (j % stages), (uint32_t)(j / stages) & 1u, kDrainTimeoutNs)) {
                    record_error(p, kErrProducerDrain);
                    break;
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA warp
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish_alloc_permit();
        ptx::tcgen05_fence_before_thread_sync();
        __syncwarp();
        ptx::tcgen05_fence_after_thread_sync();
        const uint32_t tmem_d = *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot);
        ptx::mbar_arrive(bar_tmem_alloc);          // phase 0: "TMEM allocated" (32 lanes)

        if (lane == 0) {
            int i = 0;
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                const int b = j & 1;
                const uint32_t u = (uint32_t)(j >> 1);
                // The epilogue must have read this buffer's previous tile.
                if (!wait_bounded<false>(bar_acc_empty + 8u * b, (u & 1u) ^ 1u, p.timeout_ns)) {
                    record_error(p, kErrMmaFull);
                    break;
                }
                ptx::tcgen05_fence_after_thread_sync();
                const uint32_t d = tmem_d + (uint32_t)b * kBufCols;
                for (int st = 0; st < spt; ++st, ++i) {
                    const int s = i % stages;
                    const uint32_t ph = (uint32_t)(i / stages) & 1u;
                    if (!wait_bounded<false>(bar_full + 8u * s, ph, p.timeout_ns)) {
                        record_error(p, kErrMmaFull);
                        ok = false;
                        break;
                    }
                    if (p.timeline != nullptr && (i == 0 || i == my_tiles * spt - 1))
                        p.timeline[4 * blockIdx.x + (i == 0 ? 1 : 2)] = ptx::globaltimer();
                    ptx::tcgen05_fence_after_thread_sync();
                    mma_stage<TILE_N, M_PAD, 1>(d, sbase + L.w + (uint32_t)s * w_stage_bytes,
                                                sbase + L.a + (uint32_t)s * a_stage_bytes, kbs, st == 0, 0);
                    ptx::tcgen05_commit(bar_empty + 8u * s);
                }
                ptx::tcgen05_commit(bar_acc_full + 8u * b);
            }
        }
        __syncwarp();

        // TMEM release after the epilogue's last loads: the same two-phase
        // argument as in lowm_splitk_kernel (phase 0 = the 32 arrivals above plus
        // the epilogue's first arrivals; this warp observes phase 0 before its
        // second arrival, so phase 1 = its second arrivals plus the epilogue's
        // arrivals made after its final tcgen05.wait::ld).
        if (!wait_bounded<false>(bar_tmem_alloc, 0, p.timeout_ns))
            record_error(p, kErrMmaTmemPhase0);
        ptx::mbar_arrive(bar_tmem_alloc);
        if (!wait_bounded<false>(bar_tmem_alloc, 1, p.timeout_ns))
            record_error(p, kErrMmaTmemPhase1);
        // Every MMA this CTA issued has completed: the last commit on each buffer.
        for (int b = 0; b < 2 && b < my_tiles; ++b) {
            const int last = my_tiles - 1 - ((my_tiles - 1 - b) & 1);   // last tile index with parity b
            if (!wait_bounded<false>(bar_acc_full + 8u * b, (uint32_t)(last >> 1) & 1u, kDrainTimeoutNs))
                record_error(p, kErrMmaAccDrain);
        }
        ptx::tcgen05_fence_after_thread_sync();
        if (p.probes != nullptr)
            probe_before_dealloc(p, lane, tmem_slot + kTicketOffset);
        ptx::tmem_dealloc(tmem_d, kTmemCols);
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int quarter = warp & 3;
        const int etid = threadIdx.x - kEpilogueWarp0 * 32;
        if (((p.stall_warp_mask >> warp) & 1u) && (p.stall_rank_mask == 0 || ((p.stall_rank_mask >> rank) & 1u))) {
            const uint64_t t0 = ptx::globaltimer();
            while (ptx::globaltimer() - t0 < p.stall_ns)
                ptx::nanosleep(256);
        }
        ptx::mbar_arrive(bar_tmem_alloc);          // first arrival: phase 0
        bool ok = wait_bounded<false>(bar_tmem_alloc, 0, p.timeout_ns);
        if (!ok)
            record_error(p, kErrEpiTmemPhase0);
        ptx::tcgen05_fence_after_thread_sync();
        const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot);
        ptx::griddep_wait();
        int row;
        const bool valid = tmem_row_of_thread<TILE_N>(quarter, lane, row);
        unsigned long long t_ld = 0;

        for (int j = 0; j < my_tiles; ++j) {
            const int b = j & 1;
            const uint32_t u = (uint32_t)(j >> 1);
            const int n0 = (cluster + j * clusters) * kTileN;
            if (ok && !wait_bounded<false>(bar_acc_full + 8u * b, u & 1u, p.timeout_ns)) {
                record_error(p, kErrEpiAccFull);
                ok = false;
            }
            ptx::tcgen05_fence_after_thread_sync();
            ok = __all_sync(0xffffffffu, ok);
            float acc[M_PAD];
            if (ok) {
                load_accumulator<M_PAD>(tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)b * kBufCols, acc);
            } else {
#pragma unroll
                for (int i = 0; i < M_PAD; ++i)
                    acc[i] = 0.0f;
            }
            if (p.probes != nullptr)
                t_ld = ptx::globaltimer();
            ptx::tcgen05_fence_before_thread_sync();
            ptx::mbar_arrive(bar_acc_empty + 8u * b);    // the MMA warp may overwrite this buffer

            if (SPLIT_K > 1 && rank != 0) {
                // Wait until the owner has consumed this mailbox buffer's previous tile.
                bool free_ok = wait_bounded<true>(bar_mbox_free + 8u * b, (u & 1u) ^ 1u, p.timeout_ns);
                if (!free_ok)
                    record_error(p, kErrReduce);
                ptx::fence_acquire_shared_cluster();
                if (ok && free_ok && valid && !p.drop_mailbox) {
                    const uint32_t dst = ptx::mapa_shared(
                        sbase + L.mailbox + (uint32_t)b * kSetBytes + ((rank - 1u) * kTileN + (uint32_t)row) * (M_PAD * 4u),
                        0);
                    const uint32_t rbar = ptx::mapa_shared(bar_reduce + 8u * b, 0);
#pragma unroll
                    for (int i = 0; i < M_PAD / 4; ++i)
                        ptx::st_async_v4(dst + 16u * i, rbar, acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                }
            } else {
                bool red_ok = true;
                if (SPLIT_K > 1) {
                    if (!owner_wait_mailbox(p, bar_reduce + 8u * b, u & 1u))
                        red_ok = false;
                    ptx::fence_acquire_shared_cluster();
                    if (valid && red_ok) {
                        const float *box = reinterpret_cast<const float *>(smem + L.mailbox + (uint32_t)b * kSetBytes);
#pragma unroll 1
                        for (int r = 1; r < SPLIT_K; ++r) {            // fixed rank order
                            const float4 *src =
                                reinterpret_cast<const float4 *>(box + ((r - 1) * kTileN + row) * M_PAD);
#pragma unroll
                            for (int i = 0; i < M_PAD / 4; ++i) {
                                const float4 v = src[i];
                                acc[4 * i] += v.x;
                                acc[4 * i + 1] += v.y;
                                acc[4 * i + 2] += v.z;
                                acc[4 * i + 3] += v.w;
                            }
                        }
                    }
                }
                __nv_bfloat16 *stage_out = reinterpret_cast<__nv_bfloat16 *>(smem + L.out + (uint32_t)b * kOutBytes);
                if (valid) {
#pragma unroll
                    for (int m = 0; m < M_PAD; ++m)
                        stage_out[m * kTileN + row] = __float2bfloat16_rn(acc[m]);
                    if (p.c_f32 != nullptr) {
#pragma unroll
                        for (int m = 0; m < M_PAD; ++m)
                            if (m < p.M && n0 + row < p.N)
                                p.c_f32[(size_t)m * p.N + n0 + row] = acc[m];
                    }
                }
                // Every epilogue thread has read mailbox buffer b and written its staging rows.
                ptx::named_barrier_sync(1, kEpilogueThreads);
                if (SPLIT_K > 1 && etid == 0 && j + 2 < my_tiles) {
                    // Re-arm buffer b for tile j + 2, then tell each peer it may write it.
                    ptx::mbar_arrive_expect_tx(bar_reduce + 8u * b, kSetBytes);
#pragma unroll 1
                    for (int r = 1; r < SPLIT_K; ++r)
                        ptx::mbar_arrive_remote_release_cluster(ptx::mapa_shared(bar_mbox_free + 8u * b, (uint32_t)r));
                }
                if ((p.N & 7) == 0) {
                    // 16-byte coalesced stores: row m of the tile is tile_n bf16 = tile_n / 8
                    // chunks; a partial last tile stores only the chunks below N.
                    for (int c = etid; c < p.M * (kTileN / 8); c += kEpilogueThreads) {
                        const int m = c / (kTileN / 8), ch = c % (kTileN / 8);   // 16-byte chunk ch of row m
                        if (n0 + ch * 8 < p.N) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(stage_out + m * kTileN + ch * 8);
                            *reinterpret_cast<uint4 *>(p.C + (size_t)m * p.N + n0 + ch * 8) = v;
                        }
                    }
                } else {
                    // N not a multiple of 8: rows of C are not 16-byte aligned; store elements.
                    for (int e = etid; e < p.M * kTileN; e += kEpilogueThreads) {
                        const int m = e / kTileN, col = e % kTileN;
                        if (n0 + col < p.N)
                            p.C[(size_t)m * p.N + n0 + col] = stage_out[m * kTileN + col];
                    }
                }
            }
        }
        if (p.timeline != nullptr && etid == 0)
            p.timeline[4 * blockIdx.x + 3] = ptx::globaltimer();
        if (p.probes != nullptr)
            probe_loads_done(p, t_ld, lane, tmem_slot + kTicketOffset);
        ptx::tcgen05_fence_before_thread_sync();
        ptx::mbar_arrive(bar_tmem_alloc);          // second arrival: every TMEM read of this thread is done
    }
}

}  // namespace lowm
