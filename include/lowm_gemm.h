/*
 * lowm_gemm.h -- C ABI of the GB300 (sm_103a) low-M split-K bf16 GEMM.
 *
 * The library computes
 *
 *     C[M,N] = A[M,K] . W[N,K]^T        bf16 inputs, fp32 accumulation, bf16 output
 *
 * for small M (1..128): a weight matrix W is streamed once from HBM while the
 * few activation rows A are reused by every CTA.  This is the operation of the
 * low-M split-K GEMM described in the TensorRT-LLM PR "Fix two synchronization
 * gaps in the MiniMax M3 low-M split-K GEMM" (Description; Hardware
 * verification): K is split across the CTAs of one thread-block cluster, the
 * non-owner ranks push their fp32 partial tiles into the owner's (rank 0's)
 * shared-memory mailbox with st.async + complete_tx, and rank 0 sums them in
 * rank order, converts to bf16 and stores.
 *
 * Conventions shared by every entry point:
 *   - Layouts: A row-major [M,K] (K contiguous), W row-major [N,K] (K
 *     contiguous, i.e. the K-major weight), C row-major [M,N].  All three are
 *     bf16 (IEEE binary32 upper halves), passed as plain device pointers unless
 *     the name says "host".
 *   - Ownership: the caller owns every buffer.  No entry point allocates or
 *     frees device memory.  The library keeps only process-wide state: a small
 *     cache of TMA descriptors, per-kernel attribute flags, and one device
 *     status word (a module global).
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Calls enqueue work and return; they do not synchronize
 *     (except lowm_gemm_sync_status and lowm_gemm_bf16_host, as documented).
 *   - Errors: argument checks run before anything is enqueued; a rejected call
 *     writes nothing and launches nothing.  A CUDA runtime failure maps to
 *     LOWM_ERR_CUDA.  Kernel-side timeouts (a bounded wait that gave up) are
 *     recorded in the device status word and reported by
 *     lowm_gemm_sync_status.  No C++ exception crosses this boundary.
 *   - Threads: entry points may be called from several host threads; the
 *     descriptor cache is locked internally.
 *   - Device: the current CUDA device must be compute capability 10.3
 *     (GB300); otherwise LOWM_ERR_UNSUPPORTED_ARCH.
 */
#ifndef LOWM_GEMM_H
#define LOWM_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LOWM_OK = 0,
    LOWM_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative or zero size, bad option */
    LOWM_ERR_UNSUPPORTED_SHAPE = 2,  /* a shape rule below is broken */
    LOWM_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
    LOWM_ERR_UNSUPPORTED_ARCH = 4,   /* the current device is not sm_103 */
    LOWM_ERR_CUDA = 5,               /* a CUDA runtime call failed */
    LOWM_ERR_TIMEOUT = 6             /* a kernel's bounded wait gave up (see lowm_gemm_sync_status) */
} lowm_status_t;

/*
 * A tactic: how one GEMM is tiled and launched.
 *   tile_n       output columns per CTA; the MMA's M dimension (swap-AB: N is
 *                mapped onto the tensor core's M, the tiny M onto its N): 128
 *                when N % 128 == 0, split_k <= 4 and the 128-column grid has
 *                64 CTAs to two per SM, each streaming at most 768 KiB of W
 *                unless every SM gets one (at m_pad >= 48 also: the
 *                64-column grid would not fit one CTA per SM, and split_k 2
 *                or one CTA per SM); else 64
 *   m_pad        M rounded up to the MMA's N granularity (8, 16, 32, 48, 64, 96 or 128;
 *                at least 16 for 128-column tiles); rows M..m_pad-1 are
 *                zero-filled by the TMA unit and never stored
 *   split_k      CTAs per cluster along K (1, 2, 3, 4 or 8).  K is cut into
 *                stages of kb_per_stage 64-wide blocks and rank r takes
 *                stages [r*T/split_k, (r+1)*T/split_k) of the T in all, so
 *                the ranks' shares differ by at most one stage
 *   stages       depth of the shared-memory ring between the TMA producer and the MMA warp
 *   block_k      K elements per block (64: one 128-byte swizzle row of bf16)
 *   tiles        ceil(N / tile_n) output tiles (the last may be partial)
 *   num_clusters clusters launched: `tiles` (one tile each), or fewer when
 *                persistent
 *   ctas         num_clusters * split_k
 *   smem_bytes   dynamic shared memory requested per CTA
 *   pdl          1 when launched with programmatic dependent launch
 *   persistent   1: each cluster walks tiles c, c + num_clusters, ... with a
 *                continuous TMA stream and double-buffered accumulator,
 *                mailbox and output staging (opt-in with the environment
 *                variable LOWM_PERSISTENT=1, even K splits only; every cluster
 *                then gets the same number of tiles, tiles_per_cluster)
 *   tiles_per_cluster  ceil(tiles / num_clusters)
 *   kb_per_stage 64-wide K blocks per ring stage, fetched by one 3-D TMA
 *                copy of W and one of A (the largest of 8, 4, 2, 1 that
 *                divides the rank's block count and whose two-stage ring
 *                fits the per-SM shared-memory budget, and 160 KiB of W
 *                unless one CTA per SM runs with the W promise or streams
 *                more than 512 KiB of W): a copy has
 *                a fixed per-CTA cost, so larger copies are what let one CTA
 *                stream its share of HBM
 *   mma_issuers  threads issuing tcgen05.mma per CTA: 2 for the one-tile
 *                kernel (one takes the even, the other the odd 16-wide K steps
 *                of every stage, each into its own TMEM accumulator; the
 *                epilogue adds accumulator 0 + accumulator 1), 1 for the
 *                persistent kernel.  One thread issues an MMA only every ~55
 *                cycles, so at small m_pad the issuer paces the stream.
 *   w_prefetch_stages  ring stages of W requested before the
 *                programmatic-dependency wait under
 *                LOWM_FLAG_W_BEFORE_PDL_WAIT (0 without the flag)
 *   mbox_in_ring 1: the split-K mailbox and the output staging share the
 *                owner's ring memory, which they use only after the owner's
 *                last MMA has completed (the owner then tells each peer that
 *                its mailbox is open); a CTA needs max(ring, mailbox) bytes of
 *                shared memory instead of their sum.  0: the mailbox sits
 *                after the ring; at m_pad 64 with split_k 2 the exchange is
 *                then a reduce-scatter: each rank sends the other rank its
 *                partial of the other half of the m_pad rows, adds the other
 *                rank's partial of its own half (the rank-ordered sum of two
 *                terms) and stores those rows of C.
 *   l2_prefetch_stages  stages of W the producer requests into L2 (TMA
 *                prefetch, no shared-memory destination) ahead of its newest
 *                ring load, so that one more stage of W is in flight than the
 *                ring's shared memory holds (0: none; the persistent kernel
 *                uses none)
 *   l2_before_wait_stages  without LOWM_FLAG_W_BEFORE_PDL_WAIT: stages of W
 *                requested into L2 (not into shared memory) before the
 *                programmatic-dependency wait.  A kernel that runs before
 *                this one and writes W writes through L2, so the later ring
 *                loads still read the current W; no promise is needed.  0
 *                with the flag (the ring itself is then requested early) and
 *                for the persistent kernel.
 * The pages' shipped tactic reads as (tile_n 64, m_pad 8, split_k 2, stages 10)
 * ("Fix two synchronization gaps ...", Hardware verification).
 */
typedef struct {
    int tile_n, m_pad, split_k, stages, block_k;
    int tiles, num_clusters, ctas, smem_bytes, pdl;
    int persistent, tiles_per_cluster, kb_per_stage;
    int mma_issuers, w_prefetch_stages;
    int mbox_in_ring, l2_prefetch_stages;
    int l2_before_wait_stages;
} lowm_tactic_t;

/*
 * C = A . W^T on `stream`: the low-M split-K GEMM of the PR page
 * (Description; the launch shape of Hardware verification: clusters of
 * split_k CTAs along the output columns, programmatic dependent launch on).
 *   M        1..128 (M 65..96 pads to m_pad 96, M 97..128 to 128; those
 *            shapes run split_k 1, 2, 3 or 4 with 64-column tiles, 1, 2 or 3
 *            with 128-column tiles)
 *   N        any positive value; when N is not a multiple of tile_n the last
 *            tile is partial (the TMA unit zero-fills W rows >= N and the
 *            epilogue stores only columns < N; 16-byte stores when N % 8 == 0,
 *            element stores otherwise)
 *   K        a positive multiple of 64 with K / 64 >= split_k (every rank
 *            gets a non-empty share of K, the condition the TMEM-release
 *            argument of the PR page's Description relies on)
 *   split_k  0 (let the tactic table choose), 1, 2, 3, 4 or 8
 *   A, W, C  device pointers, 16-byte aligned; C must not overlap A or W
 * Returns LOWM_OK once the kernel is enqueued.  Errors, all before anything
 * is enqueued: LOWM_ERR_INVALID_ARGUMENT (a NULL pointer, M, N or K <= 0,
 * split_k outside {0, 1, 2, 3, 4, 8}, C overlapping A or W),
 * LOWM_ERR_MISALIGNED, LOWM_ERR_UNSUPPORTED_SHAPE (a rule above, or no
 * tactic whose shared memory fits), LOWM_ERR_UNSUPPORTED_ARCH; a failed
 * launch returns LOWM_ERR_CUDA.  The result is deterministic: the same
 * arguments and tactic give the same bits on every launch.
 */
lowm_status_t lowm_gemm_bf16(const void *A, const void *W, void *C,
                             int M, int N, int K, int split_k, void *stream);

/*
 * Flags for lowm_gemm_bf16_ex.
 *
 * LOWM_FLAG_W_BEFORE_PDL_WAIT: the caller promises that W is not written by
 * the kernel that precedes this launch in the stream (true for weights).  The
 * kernel may then request its first ring of W tiles before the programmatic
 * dependent launch wait, so those loads overlap the preceding kernel's tail.
 * A and C are still touched only after the wait.  Breaking the promise gives
 * undefined results.
 */
#define LOWM_FLAG_W_BEFORE_PDL_WAIT 1u

/*
 * LOWM_FLAG_A_BEFORE_PDL_WAIT: the caller promises that A is not written by
 * the kernel that precedes this launch in the stream either (GEMMs that share
 * one input, such as projections of the same activations).  The kernel then
 * loads A without waiting for the preceding kernel; only its stores of C wait
 * for it.  It takes effect together with LOWM_FLAG_W_BEFORE_PDL_WAIT (alone,
 * W is still read after the wait, and so is A).  Breaking the promise gives
 * undefined results.
 */
#define LOWM_FLAG_A_BEFORE_PDL_WAIT 2u

/*
 * lowm_gemm_bf16 with launch flags (a bitwise OR of LOWM_FLAG_*; unknown bits
 * are rejected with LOWM_ERR_INVALID_ARGUMENT).  flags == 0 is lowm_gemm_bf16.
 */
lowm_status_t lowm_gemm_bf16_ex(const void *A, const void *W, void *C,
                                int M, int N, int K, int split_k, unsigned int flags, void *stream);

/*
 * Fill *out with the tactic lowm_gemm_bf16 would launch for these arguments
 * (host only; no device work).  Same argument rules and status codes as
 * lowm_gemm_bf16, minus the pointer checks.  The PR page runs its kernel with
 * a host-chosen tactic ("Fix two synchronization gaps ...", Hardware
 * verification: the shipped (64, 8, 2, 10) tactic, 96 clusters / 192 CTAs at
 * M4 N6144 K4096); it defines no query, and this one reports the table's
 * choice (tile, padding, split, ring, grid, shared memory) for a shape.
 */
lowm_status_t lowm_gemm_query_tactic(int M, int N, int K, int split_k, lowm_tactic_t *out);

/*
 * The tactic lowm_gemm_bf16_ex launches with these flags (LOWM_FLAG_*; unknown
 * bits are rejected with LOWM_ERR_INVALID_ARGUMENT).  The choice depends on
 * the W promise: with LOWM_FLAG_W_BEFORE_PDL_WAIT and one CTA per SM the ring
 * may fill the SM's shared memory (its first stages are requested before the
 * dependency wait); without it the ring holds at most 160 KiB of W unless a
 * CTA streams more than 512 KiB of W, and the first stages of W are
 * requested into L2 only (l2_before_wait_stages).
 * lowm_gemm_query_tactic is this call with flags 0.
 */
lowm_status_t lowm_gemm_query_tactic_ex(int M, int N, int K, int split_k, unsigned int flags, lowm_tactic_t *out);

/* A static, human-readable name for a status code (never NULL).  The pages'
 * kernel reports no errors, so this helper of the boundary has no passage
 * behind it. */
const char *lowm_status_string(lowm_status_t status);

/*
 * Synchronize `stream`, then read and clear the device status word that the
 * kernels set when a bounded wait gives up.  The pages' kernel waits without
 * a bound (the PR page's Description, item 1, notes that the missing phase-0
 * wait does not hang); this library bounds every wait on another party (2 s)
 * so that a lost arrival ends the kernel with a recorded error instead of a
 * hung GPU, and this call is how the host learns of it.  Returns LOWM_ERR_TIMEOUT if any
 * kernel since the last call recorded one (the word's bits are written to
 * *detail when detail is non-NULL), LOWM_ERR_CUDA if synchronization failed,
 * else LOWM_OK.
 */
lowm_status_t lowm_gemm_sync_status(void *stream, unsigned int *detail);

/*
 * End-to-end form for callers whose operands live in host memory: copies
 * A_host and W_host into the caller-provided device buffers A_dev and W_dev,
 * runs lowm_gemm_bf16 into C_dev, copies C_dev back into C_host, all on
 * `stream`, then synchronizes `stream`.  Host buffers should be pinned for
 * asynchronous copies; pageable memory works but serializes.  Sizes follow
 * from M, N, K (A: M*K*2 bytes, W: N*K*2, C: M*N*2).
 */
lowm_status_t lowm_gemm_bf16_host(const void *A_host, const void *W_host, void *C_host,
                                  void *A_dev, void *W_dev, void *C_dev,
                                  int M, int N, int K, int split_k, void *stream);

/*
 * Test and tuning hooks.  The race-stress method of the pages ("Fix two
 * synchronization gaps ...", Hardware verification): stall some epilogue
 * warps before their first arrival on the TMEM barrier, keep the shared
 * memory request at the kernel's footprint so another kernel can co-reside
 * on the SM, run a TMEM-allocating kernel on a second stream, and probe
 * %globaltimer at the epilogue's tcgen05.ld and the MMA warp's tcgen05.dealloc.
 *
 *   stall_warp_mask  bit w set: warp w of the CTA sleeps stall_ns: epilogue
 *                    warps (2..5) before their first TMEM-barrier arrival, the
 *                    second MMA issuer (warp 6, one-tile kernel) before its
 *                    first MMA
 *   stall_rank_mask  bit r set: only cluster ranks r stall (0 = every rank)
 *   stall_ns         stall length in nanoseconds (bounded busy sleep)
 *   full_smem        0: request the kernel's footprint (the default, which
 *                    lets another kernel co-reside on the SM); 1: request the
 *                    full 227 KiB per CTA as the pages' shipped launch does,
 *                    so nothing else can co-reside
 *   stages           0: tactic default; else the ring depth to use (>= 2)
 *   drop_mailbox     1: the non-owner ranks skip their mailbox publication, so
 *                    the owner's mailbox wait runs out (a dropped message, to
 *                    test the timeout path); the output is then undefined.
 *                    In the reduce-scatter exchange every rank skips its
 *                    publication and every rank's wait runs out.
 *                    After a mailbox wait runs out, the owner waits once more
 *                    with the same bound before it exits, so that a peer that
 *                    is only slow lands its partial tile while the owner's
 *                    shared memory still exists; a peer slower than both
 *                    bounds could still write after the owner exited, which
 *                    CUDA leaves undefined, so treat LOWM_ERR_TIMEOUT as
 *                    fatal for the outputs of the launches it reports.
 *   reduce_timeout_ns 0: default (2 s); else the bound on the owner's
 *                    mailbox wait.  Every other wait keeps its 2 s bound.
 *   probes           NULL, or device u64[3 * ctas]: per CTA (by linear CTA
 *                    index) [0] = latest %globaltimer after any epilogue
 *                    thread's last tcgen05.wait::ld, [1] = %globaltimer just
 *                    before tcgen05.dealloc, [2] = the ordering tickets the
 *                    MMA warp saw just before tcgen05.dealloc: each of the 4
 *                    epilogue warps takes one from a shared counter after its
 *                    last tcgen05.wait::ld and before its release arrival, so
 *                    4 means every epilogue load was complete when TMEM was
 *                    freed (an exact order, unlike two clock reads that can
 *                    fall in the same timer tick).  Zero-initialise before
 *                    the launch.
 *   c_f32            NULL, or device float[M*N]: the fp32 sums before the bf16
 *                    rounding (written by the owner rank)
 *   flags            launch flags as for lowm_gemm_bf16_ex (LOWM_FLAG_*)
 *   timeline         NULL, or device u64[4 * ctas]: per CTA, %globaltimer at
 *                    [0] the end of the prologue, [1] the MMA warp's first
 *                    full stage, [2] its last full stage, [3] the end of the
 *                    epilogue (a diagnostic of where a launch spends its time)
 */
typedef struct {
    unsigned int stall_warp_mask;
    unsigned int stall_rank_mask;
    unsigned int stall_ns;
    int full_smem;
    int stages;
    int drop_mailbox;
    unsigned long long reduce_timeout_ns;
    unsigned long long *probes;
    float *c_f32;
    unsigned long long *timeline;
    unsigned int flags;
} lowm_debug_opts_t;

/* lowm_gemm_bf16 with the hooks above (opts may be NULL: same as lowm_gemm_bf16). */
lowm_status_t lowm_gemm_bf16_debug(const void *A, const void *W, void *C,
                                   int M, int N, int K, int split_k, void *stream,
                                   const lowm_debug_opts_t *opts);

/*
 * The concurrent TMEM allocator of the stress method: `ctas` CTAs, each
 * allocates `ncols` TMEM columns (32..256, a power of two), writes NaN into
 * every lane of them `iters` times, frees them and exits.  It never waits on
 * another kernel.  Enqueued on `stream`.
 */
lowm_status_t lowm_tmem_hog_launch(void *stream, int ctas, int ncols, int iters);

#ifdef __cplusplus
}
#endif

#endif /* LOWM_GEMM_H */
