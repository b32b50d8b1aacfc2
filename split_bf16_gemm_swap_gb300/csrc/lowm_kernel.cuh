// The low-M split-K bf16 GEMM kernel for sm_103a:  C[M,N] = A[M,K] . W[N,K]^T.
//
// One CTA owns a tile_n-column slice of C (tile_n = 64 or 128) and 1/split_k of K.  The
// split_k CTAs of a slice form one thread-block cluster along grid x; rank 0
// of the cluster is the owner that reduces and stores.  Warp roles:
//   warp 0      TMA producer: streams W and A through a ring of `stages`
//               shared-memory stages (full/empty mbarrier pair per stage).
//               A stage holds `kb_per_stage` 64-wide K blocks: one 3-D copy of
//               W [kb_per_stage x 64 n x 64 k] and one of A [kb_per_stage x
//               m_pad x 64 k], each block a standard 128-byte-swizzled tile.
//               A copy costs about the same fixed time per CTA whatever its
//               size, so fewer, larger copies are what lets one CTA stream
//               its share of HBM bandwidth.
//   warp 1      MMA warp: allocates TMEM, issues tcgen05.mma (swap-AB: the W
//               tile is the MMA's A operand with M = tile_n, the activation
//               tile is its B operand with N = m_pad) for the even K16 steps
//               of every stage into accumulator 0, releases each stage with
//               tcgen05.commit, and frees TMEM after the epilogue's loads.
//   warp 6      second MMA issuer: the odd K16 steps of every stage into
//               accumulator 1.  One thread issues a tcgen05.mma only every
//               ~55 cycles whatever the shape (measured on GB300), which at
//               m_pad 8 makes a single issuer the pace-setter of a CTA's
//               stream; two issuers halve the time a stage is held.
//   warps 2..5  epilogue: tcgen05.ld of both fp32 accumulators, summed
//               (accumulator 0 + accumulator 1), split-K exchange through the
//               owner's shared-memory mailbox, fp32 -> bf16 and 16-byte
//               stores of C.
//
// Sources for the method ("Fix two synchronization gaps in the MiniMax M3
// low-M split-K GEMM", TensorRT-LLM PR):
//   - Description, item 1: the TMEM barrier bar_tmem_alloc with 160 arrivals
//     (32 MMA-warp lanes + 128 epilogue threads) and two phases; the fix makes
//     the MMA warp observe phase 0 before its release arrival.  (The second
//     MMA issuer does not arrive on it: it is ordered by the named-barrier
//     hand-off before its MMAs and by bar_acc before the dealloc.)
//   - Description, item 2: peers publish fp32 partials with
//     st.async ... complete_tx into rank 0's shared memory, crediting
//     bar_reduce; rank 0 waits with a relaxed cluster-scope parity wait and
//     then one fence.acquire.sync_restrict::shared::cluster.cluster.
//   - Hardware verification: the shipped tactic (64, 8, 2, 10), PDL on, the
//     stall / trimmed-request / TMEM-hog stress method and globaltimer probes.
// The cuLA PR "Fix SM90 WY input buffer reuse before WGMMA completion" gives
// the stage-release rule kept here: a stage is handed back to the producer
// only by tcgen05.commit, i.e. after the MMAs that read it have completed.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace lowm {

// Output columns per CTA (tile_n) = the MMA's M: 64 or 128, a template
// parameter of the kernels.
constexpr int kBlockK = 64;         // K elements per block (one 128-byte swizzle row of bf16)
constexpr int kMmaK = 16;           // K per tcgen05.mma of kind::f16
constexpr int kMaxKbPerStage = 8;   // K blocks per stage: 1, 2, 4 or 8
constexpr int kThreads = 224;       // lowm_splitk_kernel: 7 warps (TMA, MMA, 4 epilogue, second MMA issuer)
constexpr int kThreadsPersistent = 192;   // lowm_splitk_persistent_kernel: 6 warps, one MMA issuer
constexpr int kEpilogueWarp0 = 2;   // warps 2..5; warp % 4 covers every TMEM lane quarter once
constexpr int kMmaWarp2 = 6;        // second MMA issuer of lowm_splitk_kernel
constexpr uint32_t kMmaHandoffBarrier = 2;   // named barrier: MMA warp -> second issuer (TMEM address)
constexpr int kEpilogueThreads = 128;
__host__ __device__ constexpr uint32_t w_block_bytes(int tile_n)   // one tile_n x 64 W block
{
    return (uint32_t)tile_n * kBlockK * 2u;
}
constexpr uint32_t kTmemBarArrivals = 32 + kEpilogueThreads;
constexpr uint32_t kTicketOffset = 8;      // byte offset of the ordering-ticket counter from SmemLayout::tmem_slot
constexpr int kProbeWords = 3;             // probes per CTA: [t_ld, t_dealloc, tickets seen at dealloc]
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;     // 2 s per wait on another party
constexpr uint64_t kDrainTimeoutNs = 2000000000ull;       // 2 s for this CTA's own copies / MMAs in flight

// Bits of the device status word (which wait gave up).
enum : uint32_t {
    kErrProducerEmpty = 1u << 0,
    kErrProducerDrain = 1u << 1,
    kErrMmaFull = 1u << 2,
    kErrMmaTmemPhase0 = 1u << 3,
    kErrMmaTmemPhase1 = 1u << 4,
    kErrMmaAccDrain = 1u << 5,
    kErrEpiTmemPhase0 = 1u << 6,
    kErrEpiAccFull = 1u << 7,
    kErrReduce = 1u << 8,
    kErrMailboxOpen = 1u << 9,     // a peer's wait for the owner's "mailbox open" signal (ring-aliased mailbox)
};

struct KernelParams {
    __nv_bfloat16 *C;
    unsigned int *status;   // device status word (bits of the waits that gave up), owned by the library
    int M, N, K;
    int stages;             // ring depth
    int kb_per_stage;       // 64-wide K blocks per stage
    int kb_per_rank;        // 64-wide K blocks per cluster rank (persistent kernel: an even split)
    int stages_total;       // K / (64 * kb_per_stage): rank r of lowm_splitk_kernel takes stages
                            // [r * stages_total / split_k, (r + 1) * stages_total / split_k)
    uint32_t mbox_in_ring;  // 1: the mailbox and the output staging alias the (drained) ring
    int num_tiles;          // ceil(N / tile_n) (the persistent kernel walks them; the other kernel has one per cluster)
    uint64_t timeout_ns;    // bound on every wait for another party
    uint64_t reduce_timeout_ns;   // bound on the owner's mailbox wait
    // test hooks
    uint32_t stall_warp_mask, stall_rank_mask, stall_ns;
    uint32_t drop_mailbox;  // non-owner ranks skip their publication (the owner's wait runs out)
    uint32_t w_prefetch_stages;   // stages of W requested before the programmatic-dependency wait
                                  // (0 unless the caller promised the preceding kernel does not write W)
    uint32_t l2_prefetch_stages;  // W stages requested into L2 ahead of the newest ring load (0: none)
    uint32_t l2_before_wait_stages;   // W stages requested into L2 before the programmatic-dependency
                                      // wait (0 when the W promise requests the ring itself early)
    uint32_t a_before_wait;       // 1: the caller promised the preceding kernel does not write A either
    unsigned long long *probes;     // [kProbeWords * ctas], see lowm_debug_opts_t
    float *c_f32;
    unsigned long long *timeline;   // [4 * ctas]: prologue end, first / last full stage, epilogue end
};

// Shared-memory carve-up (byte offsets from a 1024-aligned base).  The same
// function sizes the launch on the host.
struct SmemLayout {
    uint32_t w, a, mailbox, out, bars, tmem_slot, bytes;
};

// `bufs` = 1 for the one-tile-per-cluster kernel, 2 for the persistent kernel
// (double-buffered mailbox and output staging).  `mbox_in_ring` (one-tile
// kernel only) places the mailbox, then the output staging, at the start of
// the ring instead of after it: both are used only once the ring is drained
// (the owner stages its output after its last MMA has completed, and a peer
// writes the owner's mailbox only after the owner has said so; see
// lowm_splitk_kernel), so a split-K CTA needs max(ring, mailbox + staging)
// bytes rather than their sum.
// Split-K 2 at m_pad 48 and 64 with the mailbox next to the ring reduces and
// scatters: rank q keeps rows [q m_pad / 2, (q + 1) m_pad / 2) of the tile, sends the other
// half of its partial to the other rank, sums its own half in rank order and
// stores it.  Both directions of the cluster link carry 16 KiB (128-column
// tiles) at once instead of one carrying 32 KiB, neither rank waits for the
// other's ring to drain, and the halved mailbox and staging leave room for a
// 4 x 2 ring next to them (GB300, M64 N6144 K4096: 10.66 -> 9.88 us with the W
// promise, 12.15 -> 11.43 us without; M48 10.56 -> 9.85 us).  At m_pad 32 it
// measured 9.59 -> 9.66 us with the promise (11.14 -> 10.79 without) and is
// not used.
__host__ __device__ constexpr bool reduce_scatter_of(int m_pad, int split_k, int bufs, bool mbox_in_ring)
{
    return split_k == 2 && bufs == 1 && !mbox_in_ring && (m_pad == 48 || m_pad == 64);
}

__host__ __device__ inline uint32_t ring_bytes_of(int tile_n, int m_pad, int stages, int kb_per_stage)
{
    return (uint32_t)stages * (uint32_t)kb_per_stage * (w_block_bytes(tile_n) + (uint32_t)m_pad * 128u);
}

__host__ __device__ inline SmemLayout make_smem_layout(int tile_n, int m_pad, int split_k, int stages,
                                                       int kb_per_stage, int bufs = 1, bool mbox_in_ring = false)
{
    SmemLayout L;
    uint32_t off = 0;
    L.w = off;                                            // [stages][kb_per_stage][tile_n][64 k] bf16
    off += (uint32_t)stages * (uint32_t)kb_per_stage * w_block_bytes(tile_n);
    L.a = off;                                            // [stages][kb_per_stage][m_pad][64 k]; m_pad*128 % 1024 == 0
    off += (uint32_t)stages * (uint32_t)kb_per_stage * (uint32_t)m_pad * 128u;
    // Reduce-scatter (reduce_scatter_of): each rank receives and stores half of
    // the tile's m_pad rows.
    const uint32_t rows = reduce_scatter_of(m_pad, split_k, bufs, mbox_in_ring) ? (uint32_t)m_pad / 2u
                                                                                 : (uint32_t)m_pad;
    const uint32_t mbox_bytes = (uint32_t)bufs * (uint32_t)(split_k - 1) * (uint32_t)tile_n * rows * 4u;
    const uint32_t out_bytes = (uint32_t)bufs * rows * (uint32_t)tile_n * 2u;
    if (mbox_in_ring) {
        L.mailbox = L.w;                                  // [split_k-1] slots of tile_n x m_pad fp32 (*)
        L.out = L.w + mbox_bytes;                         // [m_pad][tile_n] bf16 staging for C
        if (off < mbox_bytes + out_bytes)
            off = mbox_bytes + out_bytes;
    } else {
        L.mailbox = off;                                  // [bufs][split_k-1] slots of tile_n x m_pad fp32 (*)
        off += mbox_bytes;
        L.out = off;                                      // [bufs][m_pad][tile_n] bf16 staging for C
        off += out_bytes;
    }
    L.bars = off;                                         // full[stages], empty[stages], then per-kernel barriers
    off += (uint32_t)(2 * stages + 12) * 8u;
    L.tmem_slot = off;                                    // u32 TMEM address, then (at +8) the u32 ticket counter
    off += 16;
    L.bytes = off + 1024;                                 // slack to align the dynamic base
    return L;
}
// (*) Slot layout.  lowm_splitk_kernel stores a slot as [m_pad / 4][tile_n]
// float4, so that for one float4 index the rows of a warp are consecutive 16
// bytes: the peers' st.async writes and the owner's reads are free of bank
// conflicts.  (Rows of m_pad floats, [tile_n][m_pad], put a warp's accesses
// m_pad * 4 bytes apart: at m_pad 64 every 16-byte phase hit the same banks and
// the exchange plus reduction took ~3.6 us of a 13.3 us GEMM on GB300.)  The
// persistent kernel keeps the row layout.


// Shared-memory matrix descriptor for a K-major bf16 tile whose rows are 128
// bytes, written by TMA with 128-byte swizzling: 8-row swizzle atoms of 1024
// bytes (stride byte offset), leading byte offset unused for this layout,
// descriptor version 1, layout type 2 = SWIZZLE_128B.  Advancing the start
// address by 32 bytes selects the next 16-element K slice of the atom.
__device__ __forceinline__ uint64_t make_sw128_kmajor_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);            // start address        bits  0-13
    d |= (uint64_t)(16u >> 4) << 16;                      // leading byte offset  bits 16-29
    d |= (uint64_t)(1024u >> 4) << 32;                    // stride byte offset   bits 32-45
    d |= (uint64_t)1 << 46;                               // version              bits 46-47
    d |= (uint64_t)2 << 61;                               // SWIZZLE_128B         bits 61-63
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, shape M x N (M = tile_n, N = m_pad).
__host__ __device__ constexpr uint32_t make_idesc_bf16(int mma_m, int mma_n)
{
    return (1u << 4)                                      // D format: f32
           | (1u << 7)                                    // A format: bf16
           | (1u << 10)                                   // B format: bf16
           | ((uint32_t)(mma_n >> 3) << 17)               // N >> 3
           | ((uint32_t)(mma_m >> 4) << 24);              // M >> 4
}

__host__ __device__ constexpr uint32_t tmem_cols_for(int cols)
{
    return cols <= 32 ? 32u : (cols <= 64 ? 64u : (cols <= 128 ? 128u : (cols <= 256 ? 256u : 512u)));
}

// TMEM placement of the cta_group::1 accumulator.  M = 128: row i of D lives
// in lane i, so an epilogue warp with lane quarter q holds rows 32q..32q+31.
// M = 64: row i lives in lane 32 * (i / 16) + i % 16 (the first 16 lanes of
// each 32-lane quarter), so quarter q holds rows 16q..16q+15 in threads 0..15.
template <int TILE_N>
__device__ __forceinline__ bool tmem_row_of_thread(int quarter, int lane, int &row)
{
    if constexpr (TILE_N == 128) {
        row = 32 * quarter + lane;
        return true;
    } else {
        row = 16 * quarter + lane;
        return lane < 16;
    }
}

// Epilogue load of this warp's lane quarter: M_PAD fp32 columns, then
// tcgen05.wait::ld.
template <int M_PAD>
__device__ __forceinline__ void load_accumulator(uint32_t taddr, float (&acc)[M_PAD])
{
#pragma unroll
    for (int q = 0; q < M_PAD / 8; ++q) {
        uint32_t r[8];
        ptx::tmem_ld_32x32b_x8(taddr + 8u * q, r);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[8 * q + i] = __uint_as_float(r[i]);
    }
    ptx::tmem_wait_ld();
}

// Both accumulators' columns [0, N) for this thread's lane, with one
// tcgen05.wait::ld for all the loads: a[i] from taddr0 + i, b[i] from taddr1 + i.
template <int N>
__device__ __forceinline__ void load_accumulator_pair(uint32_t taddr0, uint32_t taddr1, float (&a)[N], float (&b)[N])
{
#pragma unroll
    for (int q = 0; q < N / 8; ++q) {
        uint32_t r0[8], r1[8];
        ptx::tmem_ld_32x32b_x8(taddr0 + 8u * q, r0);
        ptx::tmem_ld_32x32b_x8(taddr1 + 8u * q, r1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            a[8 * q + i] = __uint_as_float(r0[i]);
            b[8 * q + i] = __uint_as_float(r1[i]);
        }
    }
    ptx::tmem_wait_ld();
}

// One issuer's share of a stage's MMAs into the accumulator at tmem_d: of
// every block's 4 K16 steps, issuer q of ISSUERS takes kk = q, q + ISSUERS, ...
// `first` clears the accumulator with this issuer's first MMA of the stage.
template <int TILE_N, int M_PAD, int ISSUERS>
__device__ __forceinline__ void mma_stage(uint32_t tmem_d, uint32_t w_stage, uint32_t a_stage, int kb_per_stage,
                                          bool first, int q)
{
    constexpr uint32_t kIdesc = make_idesc_bf16(TILE_N, M_PAD);
    static_assert((kBlockK / kMmaK) % ISSUERS == 0, "issuers split the K16 steps of a block evenly");
    for (int j = 0; j < kb_per_stage; ++j) {
        const uint64_t adesc = make_sw128_kmajor_desc(w_stage + (uint32_t)j * w_block_bytes(TILE_N));
        const uint64_t bdesc = make_sw128_kmajor_desc(a_stage + (uint32_t)j * (M_PAD * 128u));
#pragma unroll
        for (int i = 0; i < kBlockK / kMmaK / ISSUERS; ++i) {
            const uint32_t kk = (uint32_t)(i * ISSUERS + q);    // +32 bytes of K per step: +2 in the encoded address
            ptx::mma_bf16_ss(tmem_d, adesc + 2u * kk, bdesc + 2u * kk, kIdesc, (first && j == 0 && i == 0) ? 0u : 1u);
        }
    }
}

template <bool kClusterScope>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    auto poll = [&]() {
        return kClusterScope ? ptx::mbar_try_wait_relaxed_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (poll())
        return true;
    // The clock is read once per 1024 polls: reading it every 32 polls cost
    // 0.1-0.5 % of a GEMM on GB300 (N6144 / N2304 / N49152 / M64 shapes);
    // every 1024 the bound stays far below the 2 s limit's resolution needs.
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        for (int i = 0; i < 1024; ++i)
            if (poll())
                return true;
        if (ptx::globaltimer() - t0 > timeout_ns)
            return false;
    }
}

__device__ __forceinline__ void record_error(const KernelParams &p, uint32_t bits)
{
    atomicOr(p.status, bits);
}

// The owner's wait for its mailbox (relaxed, cluster scope).  If it runs out,
// the error is recorded and the owner waits once more with the same bound
// before going on: a peer that is only slow then finishes its st.async writes
// into this CTA's shared memory before the CTA can exit (a write that lands
// after the owner has exited would be undefined).  The second wait also ends,
// so a peer that never writes (a dropped mailbox) costs two bounds, not a hang.
__device__ __forceinline__ bool owner_wait_mailbox(const KernelParams &p, uint32_t bar, uint32_t parity)
{
    if (wait_bounded<true>(bar, parity, p.reduce_timeout_ns))
        return true;
    record_error(p, kErrReduce);
    (void)wait_bounded<true>(bar, parity, p.reduce_timeout_ns);
    return false;
}

// A peer's wait, before its first st.async, for the owner's "mailbox open"
// arrival when the mailbox aliases the owner's ring (relaxed cluster-scope
// observation, then the acquire fence restricted to shared::cluster, as for
// the owner's mailbox wait).  Without aliasing the mailbox is always open.
__device__ __forceinline__ bool peer_wait_mailbox_open(const KernelParams &p, bool alias, uint32_t bar_open)
{
    if (!alias)
        return true;
    const bool open = wait_bounded<true>(bar_open, 0, p.timeout_ns);
    if (!open)
        record_error(p, kErrMailboxOpen);
    ptx::fence_acquire_shared_cluster();
    return open;
}

// Stress probes of the TMEM release order.  An epilogue warp calls
// probe_loads_done after its last tcgen05.wait::ld and before its release
// arrival: the latest %globaltimer of the warp goes to probes[0] and lane 0
// takes one ticket from the CTA's shared counter.  The MMA warp calls
// probe_before_dealloc after its release waits, just before tcgen05.dealloc:
// it stores %globaltimer in probes[1] and the tickets it can see in probes[2].
// The tickets make the order exact rather than a comparison of two clock
// reads: each ticket is taken before its warp's release arrival, and the MMA
// warp reads the counter after observing the phase those arrivals complete,
// so it must see all four when the protocol holds; a dealloc that could
// precede an epilogue load would see fewer.
__device__ __forceinline__ void probe_loads_done(const KernelParams &p, unsigned long long t, int lane,
                                                 uint32_t ticket_addr)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (lane == 0) {
        atomicMax(&p.probes[kProbeWords * blockIdx.x], t);
        ptx::atomic_add_shared(ticket_addr, 1u);
    }
    __syncwarp();
}

__device__ __forceinline__ void probe_before_dealloc(const KernelParams &p, int lane, uint32_t ticket_addr)
{
    if (lane == 0) {
        const unsigned long long tickets = ptx::ld_volatile_shared(ticket_addr);
        const uint64_t t = ptx::globaltimer();
        ptx::griddep_wait();                       // the probe buffer may be written by the previous kernel
        p.probes[kProbeWords * blockIdx.x + 1] = t;
        p.probes[kProbeWords * blockIdx.x + 2] = tickets;
    }
    __syncwarp();
}

// The owner's stores of one staged tile: rows m < M of [m_pad][tile_n] bf16
// staging, columns below N.  16-byte stores when N % 8 == 0 (row m of the tile
// is tile_n / 8 chunks; a partial last tile stores only the chunks below N),
// element stores otherwise (rows of C are then not 16-byte aligned).
template <int TILE_N>
__device__ __forceinline__ void store_tile(const KernelParams &p, const __nv_bfloat16 *stage_out, int n0, int etid,
                                           int m0 = 0, int m1 = -1)
{
    // Rows [m0, min(m1, M)) of C from staging rows [0, m1 - m0).
    const int rows = (m1 < 0 || m1 > p.M ? p.M : m1) - m0;
    __nv_bfloat16 *C = p.C + (size_t)m0 * p.N;
    if ((p.N & 7) == 0) {
        for (int c = etid; c < rows * (TILE_N / 8); c += kEpilogueThreads) {
            const int m = c / (TILE_N / 8), ch = c % (TILE_N / 8);   // 16-byte chunk ch of row m
            if (n0 + ch * 8 < p.N) {
                const uint4 v = *reinterpret_cast<const uint4 *>(stage_out + m * TILE_N + ch * 8);
                *reinterpret_cast<uint4 *>(C + (size_t)m * p.N + n0 + ch * 8) = v;
            }
        }
    } else {
        for (int e = etid; e < rows * TILE_N; e += kEpilogueThreads) {
            const int m = e / TILE_N, col = e % TILE_N;
            if (n0 + col < p.N)
                C[(size_t)m * p.N + n0 + col] = stage_out[m * TILE_N + col];
        }
    }
}

template <int TILE_N, int M_PAD, int SPLIT_K>
__global__ void __launch_bounds__(kThreads, 1)
    lowm_splitk_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                       const KernelParams p)
{
    static_assert(TILE_N == 64 || TILE_N == 128, "tile_n is the MMA M");
    static_assert(M_PAD % (TILE_N == 128 ? 16 : 8) == 0 && M_PAD >= 8 && M_PAD <= 128,
                  "m_pad is the MMA N: a multiple of 8 (M = 64) or 16 (M = 128), at most 128");
    constexpr int kTileN = TILE_N;
    static_assert(SPLIT_K == 1 || SPLIT_K == 2 || SPLIT_K == 3 || SPLIT_K == 4 || SPLIT_K == 8, "split_k");
    constexpr uint32_t kAcc1 = M_PAD <= 16 ? 16u : (uint32_t)M_PAD;   // column of accumulator 1
    constexpr uint32_t kTmemCols = tmem_cols_for(kAcc1 + M_PAD);
    constexpr uint32_t kSlotBytes = kTileN * M_PAD * 4u;          // one rank's fp32 partial tile

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int kbs = p.kb_per_stage;
    const bool alias = SPLIT_K > 1 && p.mbox_in_ring != 0;       // mailbox + staging in the drained ring
    constexpr bool kRsCapable = reduce_scatter_of(M_PAD, SPLIT_K, 1, false);
    const bool rs = kRsCapable && !alias;                         // reduce-scatter epilogue
    const SmemLayout L = make_smem_layout(TILE_N, M_PAD, SPLIT_K, p.stages, kbs, 1, alias);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int stages = p.stages;
    const uint32_t w_stage_bytes = (uint32_t)kbs * w_block_bytes(TILE_N);
    const uint32_t a_stage_bytes = (uint32_t)kbs * (M_PAD * 128u);
    const uint32_t stage_tx = w_stage_bytes + a_stage_bytes;
    // This rank's stages of the K range: an even share when split_k divides
    // the stage count, otherwise the first ranks take one stage fewer.
    const uint32_t rank_ = SPLIT_K > 1 ? ptx::cluster_ctarank() : 0u;
    const int s_begin = (int)(((long long)rank_ * p.stages_total) / SPLIT_K);
    const int n_stages = (int)((((long long)rank_ + 1) * p.stages_total) / SPLIT_K) - s_begin;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = rank_;
    const int n0 = (int)(blockIdx.x / SPLIT_K) * kTileN;
    const int kb0 = s_begin * kbs;

    const uint32_t bar_full = sbase + L.bars;                      // + 8 * stage
    const uint32_t bar_empty = bar_full + 8u * stages;             // + 8 * stage
    const uint32_t bar_acc = bar_full + 16u * stages;              // accumulator complete (tcgen05.commit)
    const uint32_t bar_tmem_alloc = bar_acc + 8u;                  // two phases, 160 arrivals each
    const uint32_t bar_reduce = bar_acc + 16u;                     // owner's mailbox barrier
    const uint32_t bar_reduce2 = bar_acc + 24u;                    // second half of the mailbox (two-phase)
    const uint32_t bar_open = bar_acc + 32u;                       // peers: the owner's ring is drained (alias)
    // m_pad 96 and 128: one mailbox barrier per 32-column chunk (bar_reduce,
    // bar_reduce2, bar_reduce3, and bar_reduce4 at m_pad 128), so the owner
    // reduces chunk c while the later chunks are still arriving.
    const uint32_t bar_reduce3 = bar_acc + 40u;
    const uint32_t bar_reduce4 = bar_acc + 48u;
    // m_pad 64 with the mailbox in the ring, or with split_k above 2, splits
    // each slot's float4 columns into two halves with a barrier each, so the
    // owner reduces and stages the first half while the second is still
    // arriving (GB300, M64 N6144 K4096: 11.55 -> 11.31 us; at m_pad 32 the 8
    // KiB slot gains nothing: 10.09 -> 10.14 us).
    constexpr bool kTwoPhase = SPLIT_K > 1 && M_PAD == 64;
    constexpr int kHalf4 = M_PAD / 8;                              // float4 columns in the first half
    const uint32_t tmem_slot = sbase + L.tmem_slot;

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(bar_full + 8u * s, 1);
            ptx::mbar_init(bar_empty + 8u * s, 2);        // one tcgen05.commit from each MMA issuer
        }
        ptx::mbar_init(bar_acc, 2);                        // each issuer's final commit
        ptx::mbar_init(bar_tmem_alloc, kTmemBarArrivals);
        ptx::mbar_init(bar_reduce, 1);
        ptx::mbar_init(bar_reduce2, 1);
        ptx::mbar_init(bar_open, 1);                       // one remote arrival from the owner
        ptx::mbar_init(bar_reduce3, 1);
        ptx::mbar_init(bar_reduce4, 1);
        *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot + kTicketOffset) = 0u;
        if (rs) {                          // arm this rank's half: the other rank sends half a tile
            ptx::mbar_arrive_expect_tx(bar_reduce, kSlotBytes / 2);
        } else if (SPLIT_K > 1 && rank == 0) {   // arm the mailbox: every peer sends one full partial tile
            if (M_PAD > 64) {              // one barrier per 32-column chunk (three or four)
                constexpr uint32_t kChunkTx = (SPLIT_K - 1) * kTileN * 32u * 4u;
                ptx::mbar_arrive_expect_tx(bar_reduce, kChunkTx);
                ptx::mbar_arrive_expect_tx(bar_reduce2, kChunkTx);
                ptx::mbar_arrive_expect_tx(bar_reduce3, kChunkTx);
                if (M_PAD == 128)
                    ptx::mbar_arrive_expect_tx(bar_reduce4, kChunkTx);
            } else if (kTwoPhase) {
                ptx::mbar_arrive_expect_tx(bar_reduce, (SPLIT_K - 1) * kSlotBytes / 2);
                ptx::mbar_arrive_expect_tx(bar_reduce2, (SPLIT_K - 1) * kSlotBytes / 2);
            } else {
                ptx::mbar_arrive_expect_tx(bar_reduce, (SPLIT_K - 1) * kSlotBytes);
            }
        }
        ptx::fence_mbarrier_init_cluster();
        ptx::fence_proxy_async_shared();          // the inits before this thread's own TMA copies below
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmap_w);
        ptx::prefetch_tensormap(&tmap_a);
    }
    int pre_early = 0;                             // W stages requested before the cluster wait (thread 0)
    if (SPLIT_K > 1) {
        // Peers may st.async into rank 0 only after its barriers exist.
        ptx::cluster_arrive_release();
        if (threadIdx.x == 0) {
            // Thread 0 initialised the barriers and is the TMA producer.  Between
            // its arrive and its wait it requests the first W stages (this CTA's
            // own shared memory and barriers; allowed by the caller's W
            // promise), so that a CTA placed only when the previous grid's CTAs
            // exit starts its stream ~1 us earlier.  Issued before the arrive,
            // the copies held the release arrive until they landed (GB300:
            // 12.8 us against 9.8 us at M4 N6144 K4096).
            pre_early = n_stages < stages ? n_stages : stages;
            if (pre_early > (int)p.w_prefetch_stages)
                pre_early = (int)p.w_prefetch_stages;
            const uint64_t pol_w = ptx::policy_evict_first();
            for (int i = 0; i < pre_early; ++i) {
                ptx::mbar_arrive_expect_tx(bar_full + 8u * i, stage_tx);
                ptx::tma_load_3d(sbase + L.w + (uint32_t)i * w_stage_bytes, &tmap_w, 0, n0, kb0 + i * kbs,
                                 bar_full + 8u * i, pol_w);
            }
        }
        ptx::cluster_wait_acquire();
    } else {
        __syncthreads();
    }
    if (p.timeline != nullptr && threadIdx.x == 0)
        p.timeline[4 * blockIdx.x] = ptx::globaltimer();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_first();   // W is streamed once
            const uint64_t pol_a = ptx::policy_evict_last();    // A is re-read by every CTA
            // With the caller's promise that W is not written by the preceding
            // kernel, the first w_prefetch_stages stages of W are requested
            // before the programmatic-dependency wait, overlapping that
            // kernel's tail.  A (and C, in the epilogue) are touched only after
            // the wait.
            int pre = n_stages < stages ? n_stages : stages;
            if (pre > (int)p.w_prefetch_stages)
                pre = (int)p.w_prefetch_stages;
            for (int i = pre_early; i < pre; ++i) {    // fresh ring: these stages are free (split_k 1)
                ptx::mbar_arrive_expect_tx(bar_full + 8u * i, stage_tx);
                ptx::tma_load_3d(sbase + L.w + (uint32_t)i * w_stage_bytes, &tmap_w, 0, n0, kb0 + i * kbs,
                                 bar_full + 8u * i, pol_w);
            }
            // Without the W promise, the first stages of W go to L2 (not to
            // shared memory) before the wait: L2 is where every SM's stores
            // land, so a line requested early is still the current one after
            // the wait, and the ring loads behind the wait then hit L2.
            const int l2w = pre > 0 ? 0 : (n_stages < (int)p.l2_before_wait_stages ? n_stages : (int)p.l2_before_wait_stages);
            for (int i = 0; i < l2w; ++i)
                ptx::tma_prefetch_3d(&tmap_w, 0, n0, kb0 + i * kbs);
            // A may belong to the previous kernel in the stream, unless the
            // caller promised otherwise (then only C waits, in the epilogue).
            if (!p.a_before_wait)
                ptx::griddep_wait();
            for (int i = 0; i < pre; ++i)
                ptx::tma_load_3d(sbase + L.a + (uint32_t)i * a_stage_bytes, &tmap_a, 0, 0, kb0 + i * kbs,
                                 bar_full + 8u * i, pol_a);
            // L2 prefetch: keep the W stages up to l2_prefetch_stages beyond the
            // newest ring load requested into L2, so that more of W is in
            // flight than the ring's shared memory holds.
            // (Requested before the dependency wait instead, they slowed the
            // preceding kernel's tail: 9.53 -> 11.0 us at M4 N6144 K4096.)
            const int l2pf = (int)p.l2_prefetch_stages;
            int next_pf = pre > l2w ? pre : l2w;
            while (next_pf < n_stages && next_pf < pre + l2pf) {
                ptx::tma_prefetch_3d(&tmap_w, 0, n0, kb0 + next_pf * kbs);
                ++next_pf;
            }
            int issued = pre;
            for (int i = pre; i < n_stages; ++i) {
                const int s = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (!wait_bounded<false>(bar_empty + 8u * s, ph ^ 1u, p.timeout_ns)) {
                    record_error(p, kErrProducerEmpty);
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar_full + 8u * s, stage_tx);
                const int kz = kb0 + i * kbs;
                ptx::tma_load_3d(sbase + L.w + (uint32_t)s * w_stage_bytes, &tmap_w, 0, n0, kz, bar_full + 8u * s,
                                 pol_w);
                ptx::tma_load_3d(sbase + L.a + (uint32_t)s * a_stage_bytes, &tmap_a, 0, 0, kz, bar_full + 8u * s,
                                 pol_a);
                ++issued;
                while (next_pf < n_stages && next_pf <= i + l2pf) {
                    ptx::tma_prefetch_3d(&tmap_w, 0, n0, kb0 + next_pf * kbs);
                    ++next_pf;
                }
            }
            ptx::griddep_launch_dependents();
            // No copy may still be landing in this CTA's shared memory when it exits:
            // the last load on each stage must have completed.
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
        ptx::tmem_relinquish_alloc_permit();       // let other CTAs on this SM allocate early
        ptx::tcgen05_fence_before_thread_sync();
        ptx::named_barrier_sync(kMmaHandoffBarrier, 64);   // the second issuer may now read the address
        ptx::tcgen05_fence_after_thread_sync();
        const uint32_t tmem_d = *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot);
        ptx::mbar_arrive(bar_tmem_alloc);          // phase 0: "TMEM allocated" (32 lanes)

        if (lane == 0) {
            for (int i = 0; i < n_stages; ++i) {
                const int s = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (!wait_bounded<false>(bar_full + 8u * s, ph, p.timeout_ns)) {
                    record_error(p, kErrMmaFull);
                    break;
                }
                if (p.timeline != nullptr && (i == 0 || i == n_stages - 1))
                    p.timeline[4 * blockIdx.x + (i == 0 ? 1 : 2)] = ptx::globaltimer();
                ptx::tcgen05_fence_after_thread_sync();
                mma_stage<TILE_N, M_PAD, 2>(tmem_d, sbase + L.w + (uint32_t)s * w_stage_bytes,
                                            sbase + L.a + (uint32_t)s * a_stage_bytes, kbs, i == 0, 0);
                ptx::tcgen05_commit(bar_empty + 8u * s);           // stage free once both issuers' MMAs have read it
            }
            ptx::tcgen05_commit(bar_acc);                          // accumulator 0 complete
        }
        __syncwarp();

        // TMEM release, ordered after every epilogue tcgen05.ld + wait::ld.
        // Phase 0 of bar_tmem_alloc is completed by exactly the 32 arrivals above
        // and the 128 epilogue threads' first arrivals: an epilogue thread makes
        // its second arrival only after observing phase 0, and this warp makes
        // its second arrival only after observing phase 0 too (the wait below;
        // without it, the arrival could still count toward phase 0, and the
        // parity-1 wait would then test the phase before phase 0 and return at
        // once).  Phase 1 therefore consists of these 32 second arrivals and the
        // 128 arrivals the epilogue makes after tcgen05.wait::ld, and the
        // parity-1 wait returns only when all of those have happened.
        if (!wait_bounded<false>(bar_tmem_alloc, 0, p.timeout_ns))
            record_error(p, kErrMmaTmemPhase0);
        ptx::mbar_arrive(bar_tmem_alloc);          // phase 1 (32 lanes)
        if (!wait_bounded<false>(bar_tmem_alloc, 1, p.timeout_ns))
            record_error(p, kErrMmaTmemPhase1);
        // Every MMA this CTA issued (both issuers) has completed before its
        // columns are freed (already implied on the normal path, where the
        // epilogue waited for it).
        if (!wait_bounded<false>(bar_acc, 0, kDrainTimeoutNs))
            record_error(p, kErrMmaAccDrain);
        ptx::tcgen05_fence_after_thread_sync();
        if (p.probes != nullptr)
            probe_before_dealloc(p, lane, tmem_slot + kTicketOffset);
        ptx::tmem_dealloc(tmem_d, kTmemCols);
    } else if (warp == kMmaWarp2) {
        // ------------------------------------------------------------ second MMA issuer
        // It touches TMEM only after the MMA warp has allocated it (the named
        // barrier), and the columns are freed only after its final commit has
        // arrived on bar_acc (the MMA warp's drain wait and the epilogue's
        // wait both need both commits).
        ptx::named_barrier_sync(kMmaHandoffBarrier, 64);
        ptx::tcgen05_fence_after_thread_sync();
        const uint32_t tmem_d1 = *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot) + kAcc1;
        if (((p.stall_warp_mask >> warp) & 1u) && (p.stall_rank_mask == 0 || ((p.stall_rank_mask >> rank) & 1u))) {
            const uint64_t t0 = ptx::globaltimer();     // bounded stall before its first MMA (test hook)
            while (ptx::globaltimer() - t0 < p.stall_ns)
                ptx::nanosleep(256);
        }
        if (lane == 0) {
            for (int i = 0; i < n_stages; ++i) {
                const int s = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                if (!wait_bounded<false>(bar_full + 8u * s, ph, p.timeout_ns)) {
                    record_error(p, kErrMmaFull);
                    break;
                }
                ptx::tcgen05_fence_after_thread_sync();
                mma_stage<TILE_N, M_PAD, 2>(tmem_d1, sbase + L.w + (uint32_t)s * w_stage_bytes,
                                            sbase + L.a + (uint32_t)s * a_stage_bytes, kbs, i == 0, 1);
                ptx::tcgen05_commit(bar_empty + 8u * s);
            }
            ptx::tcgen05_commit(bar_acc);                          // accumulator 1 complete
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int quarter = warp & 3;             // the TMEM lane quarter this warp may access
        const int etid = threadIdx.x - kEpilogueWarp0 * 32;
        if (((p.stall_warp_mask >> warp) & 1u) && (p.stall_rank_mask == 0 || ((p.stall_rank_mask >> rank) & 1u))) {
            const uint64_t t0 = ptx::globaltimer();     // bounded stall (test hook)
            while (ptx::globaltimer() - t0 < p.stall_ns)
                ptx::nanosleep(256);
        }
        ptx::mbar_arrive(bar_tmem_alloc);          // first arrival: phase 0
        bool ok = wait_bounded<false>(bar_tmem_alloc, 0, p.timeout_ns);
        if (!ok)
            record_error(p, kErrEpiTmemPhase0);
        ptx::tcgen05_fence_after_thread_sync();
        const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(smem + L.tmem_slot);
        ptx::griddep_wait();                       // C may belong to the previous kernel in the stream
        if (ok && !wait_bounded<false>(bar_acc, 0, p.timeout_ns)) {
            record_error(p, kErrEpiAccFull);
            ok = false;
        }
        ptx::tcgen05_fence_after_thread_sync();
        if (alias && rank == 0 && etid == 0 && ok) {
            // Every MMA of this CTA has completed (bar_acc), so no copy lands in
            // and no MMA reads the ring any more: open the mailbox that aliases
            // it to every peer (a release arrival on each peer's bar_open).
            ptx::fence_proxy_async_shared();
#pragma unroll 1
            for (int r = 1; r < SPLIT_K; ++r)
                ptx::mbar_arrive_remote_release_cluster(ptx::mapa_shared(bar_open, (uint32_t)r));
        }
        ok = __all_sync(0xffffffffu, ok);          // tcgen05.ld is warp-collective

        if constexpr (M_PAD <= 64) {
            float acc[M_PAD];
            if (ok) {
                const uint32_t lanes = (uint32_t)(32 * quarter) << 16;
                float acc1[M_PAD];
                load_accumulator_pair<M_PAD>(tmem_base + lanes, tmem_base + lanes + kAcc1, acc, acc1);
#pragma unroll
                for (int i = 0; i < M_PAD; ++i)
                    acc[i] += acc1[i];                 // fixed order: accumulator 0 + accumulator 1
            } else {
#pragma unroll
                for (int i = 0; i < M_PAD; ++i)
                    acc[i] = 0.0f;
            }
            if (p.probes != nullptr)
                probe_loads_done(p, ptx::globaltimer(), lane, tmem_slot + kTicketOffset);
            ptx::tcgen05_fence_before_thread_sync();
            ptx::mbar_arrive(bar_tmem_alloc);          // second arrival: this thread's TMEM reads are done

            int row;
            const bool valid = tmem_row_of_thread<TILE_N>(quarter, lane, row);   // row = n within the tile
            if (kRsCapable && rs) {
                if constexpr (kRsCapable) {
                    // Reduce-scatter: this rank keeps half `rank` of the m_pad rows.
                    // It sends its partial of the other half into the other rank's
                    // mailbox, then (relaxed cluster-scope wait, acquire fence) adds
                    // the other rank's partial of its own half: with two ranks the
                    // rank-ordered sum p0 + p1 is the same value in either operand
                    // order.  bf16 into staging, then its rows of C.
                    constexpr int kH4 = M_PAD / 8;                 // float4 columns per half
                    __nv_bfloat16 *stage_out = reinterpret_cast<__nv_bfloat16 *>(smem + L.out);
                    const float4 *box = reinterpret_cast<const float4 *>(smem + L.mailbox);
                    auto keep_half = [&](auto half) {
                        constexpr int H = decltype(half)::value, X = 1 - H;
                        if (ok && valid && !p.drop_mailbox) {
                            const uint32_t dst = ptx::mapa_shared(sbase + L.mailbox + 16u * (uint32_t)row, (uint32_t)X);
                            const uint32_t rbar = ptx::mapa_shared(bar_reduce, (uint32_t)X);
#pragma unroll
                            for (int i = 0; i < kH4; ++i)
                                ptx::st_async_v4(dst + 16u * kTileN * i, rbar, acc[4 * (X * kH4 + i)],
                                                 acc[4 * (X * kH4 + i) + 1], acc[4 * (X * kH4 + i) + 2],
                                                 acc[4 * (X * kH4 + i) + 3]);
                        }
                        bool okh = ok;
                        if (!owner_wait_mailbox(p, bar_reduce, 0))
                            okh = false;
                        ptx::fence_acquire_shared_cluster();
                        if (valid) {
                            if (okh) {
#pragma unroll
                                for (int i = 0; i < kH4; ++i) {
                                    const float4 v = box[i * kTileN + row];
                                    acc[4 * (H * kH4 + i)] += v.x;
                                    acc[4 * (H * kH4 + i) + 1] += v.y;
                                    acc[4 * (H * kH4 + i) + 2] += v.z;
                                    acc[4 * (H * kH4 + i) + 3] += v.w;
                                }
                            }
#pragma unroll
                            for (int m = 0; m < M_PAD / 2; ++m)
                                stage_out[m * kTileN + row] = __float2bfloat16_rn(acc[H * (M_PAD / 2) + m]);
                            if (p.c_f32 != nullptr) {
#pragma unroll
                                for (int m = H * (M_PAD / 2); m < (H + 1) * (M_PAD / 2); ++m)
                                    if (m < p.M && n0 + row < p.N)
                                        p.c_f32[(size_t)m * p.N + n0 + row] = acc[m];
                            }
                        }
                        ptx::named_barrier_sync(1, kEpilogueThreads);
                        store_tile<kTileN>(p, stage_out, n0, etid, H * (M_PAD / 2), (H + 1) * (M_PAD / 2));
                    };
                    if (rank == 0)
                        keep_half(std::integral_constant<int, 0>{});
                    else
                        keep_half(std::integral_constant<int, 1>{});
                    if (p.timeline != nullptr && etid == 0)
                        p.timeline[4 * blockIdx.x + 3] = ptx::globaltimer();
                }
            } else if (SPLIT_K > 1 && rank != 0) {
                // Non-owner: publish the partial tile into rank 0's mailbox slot (rank - 1).
                const bool open = peer_wait_mailbox_open(p, alias, bar_open);
                if (ok && open && valid && !p.drop_mailbox) {
                    const uint32_t dst = ptx::mapa_shared(
                        sbase + L.mailbox + (rank - 1u) * kSlotBytes + 16u * (uint32_t)row, 0);
                    const uint32_t rbar = ptx::mapa_shared(bar_reduce, 0);
                    const uint32_t rbar2 = kTwoPhase ? ptx::mapa_shared(bar_reduce2, 0) : rbar;
#pragma unroll
                    for (int i = 0; i < M_PAD / 4; ++i)          // slot layout [m_pad / 4][tile_n] float4
                        ptx::st_async_v4(dst + 16u * kTileN * i, (kTwoPhase && i >= kHalf4) ? rbar2 : rbar, acc[4 * i],
                                         acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                }
                if (p.timeline != nullptr && etid == 0)
                    p.timeline[4 * blockIdx.x + 3] = ptx::globaltimer();
            } else if constexpr (kTwoPhase) {
                // Owner, two-phase: per half, the relaxed cluster-scope wait and the
                // acquire fence, then the rank-ordered sum of that half's columns
                // (each element's order is the one-phase order), bf16 into staging.
                __nv_bfloat16 *stage_out = reinterpret_cast<__nv_bfloat16 *>(smem + L.out);
                const float4 *box = reinterpret_cast<const float4 *>(smem + L.mailbox);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    bool okh = ok;
                    if (!owner_wait_mailbox(p, h == 0 ? bar_reduce : bar_reduce2, 0))
                        okh = false;
                    ptx::fence_acquire_shared_cluster();
                    if (valid) {
                        if (okh) {
#pragma unroll 1
                            for (int r = 1; r < SPLIT_K; ++r) {        // fixed rank order
                                const float4 *src = box + (r - 1) * (kSlotBytes / 16) + row;
#pragma unroll
                                for (int i = h * kHalf4; i < (h + 1) * kHalf4; ++i) {
                                    const float4 v = src[i * kTileN];
                                    acc[4 * i] += v.x;
                                    acc[4 * i + 1] += v.y;
                                    acc[4 * i + 2] += v.z;
                                    acc[4 * i + 3] += v.w;
                                }
                            }
                        }
#pragma unroll
                        for (int m = h * (M_PAD / 2); m < (h + 1) * (M_PAD / 2); ++m)
                            stage_out[m * kTileN + row] = __float2bfloat16_rn(acc[m]);
                        if (p.c_f32 != nullptr) {
#pragma unroll
                            for (int m = h * (M_PAD / 2); m < (h + 1) * (M_PAD / 2); ++m)
                                if (m < p.M && n0 + row < p.N)
                                    p.c_f32[(size_t)m * p.N + n0 + row] = acc[m];
                        }
                    }
                }
                ptx::named_barrier_sync(1, kEpilogueThreads);
                store_tile<kTileN>(p, stage_out, n0, etid);
                if (p.timeline != nullptr && etid == 0)
                    p.timeline[4 * blockIdx.x + 3] = ptx::globaltimer();
            } else {
                if (SPLIT_K > 1) {
                    // Owner: relaxed cluster-scope observation of the mailbox phase,
                    // then one acquire fence restricted to shared::cluster memory.
                    if (!owner_wait_mailbox(p, bar_reduce, 0))
                        ok = false;
                    ptx::fence_acquire_shared_cluster();
                    if (valid && ok) {
                        const float4 *box = reinterpret_cast<const float4 *>(smem + L.mailbox);
#pragma unroll 1
                        for (int r = 1; r < SPLIT_K; ++r) {            // fixed rank order
                            const float4 *src = box + (r - 1) * (kSlotBytes / 16) + row;
#pragma unroll
                            for (int i = 0; i < M_PAD / 4; ++i) {
                                const float4 v = src[i * kTileN];
                                acc[4 * i] += v.x;
                                acc[4 * i + 1] += v.y;
                                acc[4 * i + 2] += v.z;
                                acc[4 * i + 3] += v.w;
                            }
                        }
                    }
                }
                if constexpr (M_PAD == 8) {
                    // m_pad 8: each thread stores its column's (at most 8) rows
                    // from registers.  The valid lanes of a warp hold consecutive
                    // columns, so every row is one contiguous 32- or 64-byte
                    // segment per warp, and the staging round trip and the
                    // 128-thread barrier disappear (GB300: 9.93 -> 9.81 us at
                    // M4 N6144 K4096, 10.52 -> 10.31 us at M4 N2304 K12288 split_k
                    // 4; at m_pad 16 and 32 staging measured as fast or faster).
                    if (valid && n0 + row < p.N) {
#pragma unroll
                        for (int m = 0; m < M_PAD; ++m)
                            if (m < p.M)
                                p.C[(size_t)m * p.N + n0 + row] = __float2bfloat16_rn(acc[m]);
                        if (p.c_f32 != nullptr) {
#pragma unroll
                            for (int m = 0; m < M_PAD; ++m)
                                if (m < p.M)
                                    p.c_f32[(size_t)m * p.N + n0 + row] = acc[m];
                        }
                    }
                } else {
                    __nv_bfloat16 *stage_out = reinterpret_cast<__nv_bfloat16 *>(smem + L.out);
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
                    ptx::named_barrier_sync(1, kEpilogueThreads);
                    store_tile<kTileN>(p, stage_out, n0, etid);
                }
                if (p.timeline != nullptr && etid == 0)
                    p.timeline[4 * blockIdx.x + 3] = ptx::globaltimer();
            }
        } else {
            // m_pad 96 and 128: two such accumulators do not fit in registers,
            // so the epilogue works in 32-column chunks.  Each chunk of the mailbox
            // has its own barrier: a peer credits chunk c's barrier with its
            // chunk-c stores, and the owner waits for chunk c only when it
            // reduces it, while the later chunks are still arriving.  Every
            // thread makes its second (TMEM-release) arrival only after its last
            // chunk's tcgen05.wait::ld.
            constexpr int kCh = 32;
            static_assert(M_PAD == 3 * kCh || M_PAD == 4 * kCh, "one mailbox barrier per 32-column chunk");
            const uint32_t lanes = (uint32_t)(32 * quarter) << 16;
            int row;
            const bool valid = tmem_row_of_thread<TILE_N>(quarter, lane, row);   // row = n within the tile
            const bool owner = !(SPLIT_K > 1 && rank != 0);
            __nv_bfloat16 *stage_out = reinterpret_cast<__nv_bfloat16 *>(smem + L.out);
            const float4 *box = reinterpret_cast<const float4 *>(smem + L.mailbox);
            uint32_t dst = 0;
            bool open = true;
            if (!owner) {
                open = peer_wait_mailbox_open(p, alias, bar_open);
                dst = ptx::mapa_shared(sbase + L.mailbox + (rank - 1u) * kSlotBytes + 16u * (uint32_t)row, 0);
            }
#pragma unroll 1
            for (int c0 = 0; c0 < M_PAD; c0 += kCh) {
                const int c = c0 / kCh;
                const uint32_t bar_c = c == 0 ? bar_reduce : c == 1 ? bar_reduce2 : c == 2 ? bar_reduce3 : bar_reduce4;
                float acc[kCh];
                if (ok) {
                    float acc1[kCh];
                    load_accumulator_pair<kCh>(tmem_base + lanes + (uint32_t)c0,
                                               tmem_base + lanes + kAcc1 + (uint32_t)c0, acc, acc1);
#pragma unroll
                    for (int i = 0; i < kCh; ++i)
                        acc[i] += acc1[i];             // fixed order: accumulator 0 + accumulator 1
                } else {
#pragma unroll
                    for (int i = 0; i < kCh; ++i)
                        acc[i] = 0.0f;
                }
                if (!owner) {
                    if (ok && open && valid && !p.drop_mailbox) {
                        const uint32_t rbar = ptx::mapa_shared(bar_c, 0);
#pragma unroll
                        for (int i = 0; i < kCh / 4; ++i)          // slot layout [m_pad / 4][tile_n] float4
                            ptx::st_async_v4(dst + 16u * kTileN * (uint32_t)(c0 / 4 + i), rbar, acc[4 * i],
                                             acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                    }
                } else {
                    bool okc = ok;
                    if (SPLIT_K > 1) {
                        // Relaxed cluster-scope observation of chunk c, then the
                        // acquire fence restricted to shared::cluster.
                        if (!owner_wait_mailbox(p, bar_c, 0))
                            okc = false;
                        ptx::fence_acquire_shared_cluster();
                    }
                    if (valid && SPLIT_K > 1 && okc) {
#pragma unroll 1
                        for (int r = 1; r < SPLIT_K; ++r) {    // fixed rank order
                            const float4 *src = box + (r - 1) * (kSlotBytes / 16) + (c0 / 4) * kTileN + row;
#pragma unroll
                            for (int i = 0; i < kCh / 4; ++i) {
                                const float4 v = src[i * kTileN];
                                acc[4 * i] += v.x;
                                acc[4 * i + 1] += v.y;
                                acc[4 * i + 2] += v.z;
                                acc[4 * i + 3] += v.w;
                            }
                        }
                    }
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < kCh; ++i)
                            stage_out[(c0 + i) * kTileN + row] = __float2bfloat16_rn(acc[i]);
                        if (p.c_f32 != nullptr) {
#pragma unroll
                            for (int i = 0; i < kCh; ++i)
                                if (c0 + i < p.M && n0 + row < p.N)
                                    p.c_f32[(size_t)(c0 + i) * p.N + n0 + row] = acc[i];
                        }
                    }
                }
            }
            if (p.probes != nullptr)
                probe_loads_done(p, ptx::globaltimer(), lane, tmem_slot + kTicketOffset);
            ptx::tcgen05_fence_before_thread_sync();
            ptx::mbar_arrive(bar_tmem_alloc);          // second arrival: this thread's TMEM reads are done
            if (owner) {
                ptx::named_barrier_sync(1, kEpilogueThreads);
                store_tile<kTileN>(p, stage_out, n0, etid);
            }
            if (p.timeline != nullptr && etid == 0)
                p.timeline[4 * blockIdx.x + 3] = ptx::globaltimer();
        }
    }
}

}  // namespace lowm
