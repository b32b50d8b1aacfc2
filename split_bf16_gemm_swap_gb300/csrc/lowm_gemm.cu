// Host side of the C ABI in include/lowm_gemm.h: argument checks, the tactic
// table, TMA descriptor encoding (cached), and the cluster + PDL launch.
//
// Launch shape ("Fix two synchronization gaps in the MiniMax M3 low-M split-K
// GEMM", TensorRT-LLM PR, Hardware verification): ceil(N / tile_n) clusters of split_k
// CTAs, programmatic dependent launch on, cluster dimension split_k along grid
// x.  The host also guarantees the non-empty K loop that the PR's analysis of
// the TMEM race relies on (Description, item 1): K must be a positive
// multiple of split_k * 64.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/lowm_gemm.h"
#include "lowm_kernels.h"

namespace lowm {

// The device status word: kernels set bits of the waits that gave up (through
// the pointer in their parameters); lowm_gemm_sync_status reads and clears it.
__device__ unsigned int g_lowm_status;

// The concurrent TMEM allocator of the stress method: allocate, fill with NaN,
// free.  128 threads; never waits on another kernel.
__global__ void __launch_bounds__(128) tmem_hog_kernel(int ncols, int iters)
{
    __shared__ uint32_t slot;
    const int warp = threadIdx.x >> 5;
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(&slot), (uint32_t)ncols);
        ptx::tmem_relinquish_alloc_permit();
    }
    ptx::tcgen05_fence_before_thread_sync();
    __syncthreads();
    ptx::tcgen05_fence_after_thread_sync();
    const uint32_t base = slot + ((uint32_t)(32 * warp) << 16);
    const uint32_t nan8[8] = {0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u,
                              0x7fc00000u, 0x7fc00000u, 0x7fc00000u, 0x7fc00000u};
    for (int it = 0; it < iters; ++it)
        for (int c = 0; c < ncols; c += 8)
            ptx::tmem_st_32x32b_x8(base + (uint32_t)c, nan8);
    ptx::tmem_wait_st();
    ptx::tcgen05_fence_before_thread_sync();
    __syncthreads();
    ptx::tcgen05_fence_after_thread_sync();
    if (warp == 0)
        ptx::tmem_dealloc(slot, (uint32_t)ncols);
}

}  // namespace lowm

namespace {

using lowm::KernelFn;
using lowm::KernelParams;
using lowm::SmemLayout;

constexpr int kMaxSmemPerCta = 232448;     // 227 KiB opt-in dynamic shared memory per CTA
constexpr int kSmemPerSm = 233472;         // 228 KiB per SM
constexpr int kSmemReservedPerCta = 1024;  // the runtime keeps 1 KiB per resident CTA

// ------------------------------------------------------------------ driver entry point
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// ------------------------------------------------------------------ device checks
struct DeviceInfo {
    bool checked = false;
    bool ok = false;
    int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

lowm_status_t check_device(int *sms_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return LOWM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.checked) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return LOWM_ERR_CUDA;
        d.ok = (major == 10 && minor == 3);
        d.sms = sms;
        d.checked = true;
    }
    if (sms_out)
        *sms_out = d.sms;
    return d.ok ? LOWM_OK : LOWM_ERR_UNSUPPORTED_ARCH;
}

// ------------------------------------------------------------------ tactics
int env_int(const char *name, int dflt)
{
    const char *v = std::getenv(name);
    return v && *v ? std::atoi(v) : dflt;
}

int m_pad_of(int M)
{
    return M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : M <= 48 ? 48 : M <= 64 ? 64 : M <= 96 ? 96 : 128;
}

int footprint(int tile_n, int m_pad, int split_k, int stages, int kbs, int bufs, bool alias = false)
{
    return (int)lowm::make_smem_layout(tile_n, m_pad, split_k, stages, kbs, bufs, alias).bytes;
}

// May a stage of `kbs` K blocks tile a K of `kb_total` blocks split `split_k`
// ways?  kbs must divide the K blocks, every rank must get at least one stage,
// and when split_k divides the blocks evenly the ranks' shares stay equal.
bool kbs_tiles_k(int kbs, int kb_total, int split_k)
{
    if (kb_total % kbs != 0 || kb_total / kbs < split_k)
        return false;
    if (kb_total % split_k == 0 && (kb_total / split_k) % kbs != 0)
        return false;
    return true;
}

// Ring shape (K blocks per stage x stages) for a launch of `ctas` CTAs on
// `sms` SMs.  From measurements on GB300 (M4 N6144/2304/49152, M16 K32768):
//   - every copy costs a fixed per-CTA time, so blocks per copy matter most;
//   - a grid that does not fit on the GPU at once wants several small CTAs per
//     SM (their prologues and epilogues overlap each other's streams): three
//     per SM without clusters, five with them;
//   - with several CTAs per SM, rings holding more than ~160 KiB of W per CTA
//     gain nothing (W bytes: the A tiles in the ring come from L2; at m_pad
//     128 an A block is twice a 64-column W block, and counting it would cap
//     that ring at 2 x 2 blocks where 4 x 2 measured 15.8 against 17.1 us at
//     M128 N6144 K4096); with one CTA per SM and the W promise, or a long
//     stream per CTA, the ring may fill the SM (below).
// Hence: budget shared memory for ceil(ctas / sms) CTAs per SM when that is at
// most 4 (the whole grid resident at once), else for 3 (split_k 1) or 5; take
// the most blocks per copy (8, 4, 2, 1, tiling K) whose 2-stage ring fits,
// then the most stages that fit.  LOWM_KB_PER_STAGE and LOWM_STAGES override
// (tuning).
struct Ring {
    int kbs, stages;
};

constexpr int kMaxRingBytes = 160 * 1024;     // W bytes per ring when several CTAs share an SM

Ring choose_ring(int tile_n, int m_pad, int split_k, int kb_total, int ctas, int sms, int bufs, bool alias = false,
                 bool deep = false)
{
    const int per_sm_one_wave = (ctas + std::max(1, sms) - 1) / std::max(1, sms);
    const int per_sm = per_sm_one_wave <= 4 ? std::max(1, per_sm_one_wave) : (split_k == 1 ? 3 : 5);
    const int budget = std::min(kMaxSmemPerCta, kSmemPerSm / per_sm - kSmemReservedPerCta);
    // One CTA per SM and a deep ring allowed (`deep`: the caller's W promise,
    // under which the first ring of W is requested before the dependency
    // wait, or a long stream per CTA): the ring may take all of the SM's
    // shared memory (a 128-column M4 N6144 K4096 CTA with a 4 x 3 ring, 192
    // KiB of W, measured 8.90 us against 9.57 us with the 4 x 2 ring the 160
    // KiB cap allows; without the promise, M4 N2304 K12288 split_k 4 on 128
    // columns, 768 KiB of W per CTA: 11.50 us against 12.12 us).  Short
    // streams without the promise measured slower with the deeper rings (4 x 3
    // 11.17 against 4 x 2 10.67 us; M4 N2304 K12288 on 64 columns 8 x 3 12.13
    // against 8 x 2 11.67 us), so the cap stays there.
    const int cap = (per_sm == 1 && deep) ? kMaxSmemPerCta : kMaxRingBytes;
    int force_kbs = env_int("LOWM_KB_PER_STAGE", 0);
    if (force_kbs != 1 && force_kbs != 2 && force_kbs != 4 && force_kbs != 8)
        force_kbs = 0;
    if (force_kbs && !kbs_tiles_k(force_kbs, kb_total, split_k))
        force_kbs = 0;                                 // a forced value that does not tile K is ignored
    const int force_st = env_int("LOWM_STAGES", 0);
    auto ring_bytes = [&](int kbs, int st) { return st * kbs * (int)lowm::w_block_bytes(tile_n); };   // W bytes
    int kbs = 1;
    if (force_kbs) {
        kbs = force_kbs;
    } else {
        for (int b = 8; b >= 1; b /= 2)
            if (kbs_tiles_k(b, kb_total, split_k) && footprint(tile_n, m_pad, split_k, 2, b, bufs, alias) <= budget &&
                ring_bytes(b, 2) <= cap) {
                kbs = b;
                break;
            }
    }
    int st = 2;
    if (force_st >= 2) {
        st = force_st;
    } else {
        while (st < 32 && footprint(tile_n, m_pad, split_k, st + 1, kbs, bufs, alias) <= budget &&
               ring_bytes(kbs, st + 1) <= cap)
            ++st;
    }
    return Ring{kbs, st};
}

// K is split in whole stages: every rank needs at least one 64-wide K block.
bool shape_ok(int M, int N, int K, int split_k)
{
    return M >= 1 && M <= 128 && N > 0 && K > 0 && K % lowm::kBlockK == 0 && K / lowm::kBlockK >= split_k;
}

// Tile width (the MMA's M), given the split.  128 columns when N is a
// multiple of 128, the split is at most 4, and the 128-column grid
//   - has at least 64 CTAs (enough concurrent streams to fill HBM) and at
//     most two per SM,
//   - streams at most 768 KiB of W per CTA or has a CTA on every SM,
//   - and, at m_pad 48 and above, replaces a 64-column grid that would not
//     fit one CTA per SM, with split_k 2 or one CTA per SM (the m_pad 64
//     mailbox of three 128-column partials leaves too small a ring);
// 64 columns otherwise.  Measured on GB300 with the W promise, 64 -> 128
// columns: N6144 K4096 split_k 2 M4 10.14 -> 9.43 us (M32 10.32 -> 9.59, M128
// 15.8 -> 14.08); split_k 4 9.72 -> 9.21; N4096 K4096 split_k 2 7.36 -> 6.79;
// N2048 K8192 split_k 4 7.62 -> 7.15; N3072 K8192 split_k 4 10.39 -> 8.87;
// N2304 K12288 split_k 4 9.99 -> 9.76 (M16 10.17 -> 10.04); M16 N6144 K32768
// split_k 4 64.2 -> 63.0; N6144 K16384 split_k 4 33.45 -> 32.72; M64 N8192
// K12288 split_k 2 34.36 -> 32.95.  Against: fewer than 64 CTAs (N2304 K12288
// split_k 2, 36 CTAs: 11.96 -> 15.77), more than two per SM (N49152 K4096:
// 61.1 -> 67.1), long streams on few CTAs (N8192 K8192 split_k 1, 64 CTAs of
// 2 MiB: 21.6 -> 25.3; N8192 K4096 split_k 1: 11.1 -> 12.4), split_k 8 (its
// seven 128-column partials take the owner's cluster link: N2304 13.1 ->
// 15.0), m_pad 64 at split_k 4 with two CTAs per SM (M64 N6144 K4096 17.4 ->
// 21.1) and m_pad 64 where the 64-column grid fits (M64 N2304 K12288 split_k
// 4 12.47 -> 13.84).  At m_pad 8 a 128-column tile pads the MMA's N to 16
// (zero rows from the TMA unit, no extra HBM bytes).  LOWM_TILE_N = 64 / 128
// overrides when the shape allows it (tuning).
constexpr int kMinStreams = 64;                          // CTAs that keep HBM busy
constexpr double kLongStreamBytes = 768.0 * 1024.0;      // W per 128-column CTA below one CTA per SM
constexpr double kShortStreamBytes = 512.0 * 1024.0;     // W per CTA the auto split aims at

int choose_tile_n(int M, int N, int K, int split_k, int sms)
{
    const int force = env_int("LOWM_TILE_N", 0);
    if (force == 128 && N >= 128)
        return 128;
    if (force == 64)
        return 64;
    if (N % 128 != 0 || split_k > 4)
        return 64;
    const long long c64 = (long long)((N + 63) / 64) * split_k, c128 = (long long)(N / 128) * split_k;
    const double per_cta = 2.0 * N * (double)K / (double)c128;
    const bool wide_pad = m_pad_of(M) >= 48;
    const bool ok = c128 >= kMinStreams && c128 <= 2LL * sms && (per_cta <= kLongStreamBytes || c128 >= sms) &&
                    (!wide_pad || (c64 > sms && (split_k <= 2 || c128 <= sms)));
    return ok ? 128 : 64;
}

int m_pad_for(int M, int tile_n)
{
    const int mp = m_pad_of(M);
    return tile_n == 128 && mp < 16 ? 16 : mp;          // MMA M = 128 needs N a multiple of 16
}

// The split-K mailbox shares the drained ring (see make_smem_layout) for
// split_k 3 and for m_pad 96 and 128, whose 24-64 KiB slots would otherwise take the
// ring's room (M128 N6144 K4096 split_k 2 on 128-column tiles: 14.4 us
// against 16.4 us with the mailbox next to the ring), and otherwise whenever
// sharing lets the ring hold more W (make_tactic compares both layouts; M4
// N6144 K4096: a 4 x 3 ring, 8.90 us, against 4 x 2, 9.57 us).  At m_pad 64
// with split_k 2 the separate mailbox is the reduce-scatter one, half the
// size, and already fits the 4 x 2 ring (9.88 us against 10.66 us for the
// same ring with the mailbox inside it).  LOWM_MBOX_IN_RING = 0 / 1
// overrides (tuning).  Returns 1 / 0 when the choice is fixed, -1 when the
// ring sizes decide.
int forced_alias(int m_pad, int split_k)
{
    if (split_k == 1)
        return 0;
    const int force = env_int("LOWM_MBOX_IN_RING", -1);
    if (force == 0 || force == 1)
        return force;
    return (split_k == 3 || m_pad > 64) ? 1 : -1;
}

bool choose_alias(int m_pad, int split_k)
{
    return forced_alias(m_pad, split_k) == 1;
}

KernelFn kernel_for(int tile_n, int m_pad, int sk, bool persistent);

// A split whose kernel instance exists, whose K loop is non-empty and even,
// and whose mailbox fits next to (or inside) a two-stage ring.
bool split_usable(int M, int N, int K, int sk, int sms)
{
    if (K % (sk * lowm::kBlockK) != 0)
        return false;
    const int tile_n = choose_tile_n(M, N, K, sk, sms);
    const int mp = m_pad_for(M, tile_n);
    return kernel_for(tile_n, mp, sk, false) &&
           footprint(tile_n, mp, sk, 2, 1, 1, choose_alias(mp, sk)) <= kMaxSmemPerCta;
}

// split_k = 0.  With N a multiple of 128: the smallest split on 128-column
// tiles (by the rule above) with at most 512 KiB of W per CTA (N6144 K4096:
// split_k 2, 96 CTAs, 8.8 us against 9.2 us at split_k 4; N4096 K4096:
// split_k 2, 64 CTAs, 6.79 against 7.25 us; N8192 K4096: split_k 2, 11.1
// against 12.4 us at split_k 1), else the largest such split for a long K (M16
// N6144 K32768: split_k 4, 192 CTAs, 63.0 us against 67.1 us at split_k 2).
// Otherwise the smallest split of 64-column tiles that fills 90 % of the SMs
// (M4 N2304 K12288 on 64 columns: split_k 4 on 144 CTAs, 10.07 us, against
// 11.08 us at split_k 8), stopping at 4 once that gives 64 CTAs: clusters of
// 8 measured slowest.  The K loop stays non-empty and the mailbox fits.
int choose_split_k(int M, int N, int K, int sms)
{
    if (N % 128 == 0) {
        const int tiles128 = N / 128;
        int longest = 0;
        for (int sk = 1; sk <= 4; sk *= 2) {
            const long long c = (long long)tiles128 * sk;
            if (c > 2LL * sms || !split_usable(M, N, K, sk, sms))
                break;
            if (c < kMinStreams || choose_tile_n(M, N, K, sk, sms) != 128)
                continue;
            if (2.0 * N * (double)K / (double)c <= kShortStreamBytes)
                return sk;
            longest = sk;
        }
        if (longest)
            return longest;
    }
    const int tiles64 = (N + 63) / 64;
    int best = 0;
    for (int sk = 1; sk <= 8; sk *= 2) {
        if (!split_usable(M, N, K, sk, sms))
            break;
        best = sk;
        if (10LL * tiles64 * sk >= 9LL * sms || (sk == 4 && tiles64 * sk >= kMinStreams))
            break;
    }
    return best;
}

// ------------------------------------------------------------------ kernels
KernelFn kernel_for(int tile_n, int m_pad, int sk, bool persistent)
{
    if (persistent && sk == 3)
        return nullptr;                                 // the persistent schedule splits K evenly (1, 2, 4, 8)
    if (m_pad == 128)
        return persistent ? nullptr : lowm::kernel_mpad128(tile_n, sk);
    if (m_pad == 96)
        return persistent ? nullptr : lowm::kernel_mpad96(tile_n, sk);
    if (m_pad == 48)
        return persistent ? nullptr : lowm::kernel_mpad48(tile_n, sk);
    if (tile_n == 64)
        return lowm::kernel_tile64(m_pad, sk, persistent);
    if (tile_n == 128)
        return lowm::kernel_tile128(m_pad, sk, persistent);
    return nullptr;
}

// Device address of the status word on the current device (looked up once per device).
unsigned int *status_word()
{
    static std::mutex mu;
    static unsigned int *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, lowm::g_lowm_status) != cudaSuccess)
            return nullptr;
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

lowm_status_t prepare_kernel(KernelFn fn)
{
    // Opt every instance into the largest request once per device.
    static std::mutex mu;
    static std::unordered_map<long long, bool> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return LOWM_ERR_CUDA;
    const long long key = (long long)reinterpret_cast<uintptr_t>(fn) * 64 + dev;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(key))
        return LOWM_OK;
    if (cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxSmemPerCta) != cudaSuccess)
        return LOWM_ERR_CUDA;
    done[key] = true;
    return LOWM_OK;
}

// Clusters of `split_k` CTAs that fit on the GPU at once with `smem` bytes
// each: the occupancy API when a usable device is current, else the per-SM
// arithmetic (shared memory and threads).
int resident_clusters(int tile_n, int m_pad, int split_k, int smem, int sms, bool persistent, bool have_device)
{
    const int threads = persistent ? lowm::kThreadsPersistent : lowm::kThreads;
    const int per_sm = std::min(kSmemPerSm / (smem + kSmemReservedPerCta), 2048 / threads);
    const int formula = sms * per_sm / split_k;
    if (!have_device)
        return formula;
    KernelFn fn = kernel_for(tile_n, m_pad, split_k, persistent);
    if (!fn || prepare_kernel(fn) != LOWM_OK)
        return formula;
    static std::mutex mu;
    static std::unordered_map<long long, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const long long key = (((long long)reinterpret_cast<uintptr_t>(fn) * 64 + dev) * 262144) + smem;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end())
            return it->second;
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(split_k * 1024), 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)split_k;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(fn), &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = formula;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = n;
    return n;
}

lowm_status_t make_tactic(int M, int N, int K, int split_k, int sms, bool have_device, unsigned flags, int stages_override,
                          int full_smem, lowm_tactic_t *t)
{
    if (M <= 0 || N <= 0 || K <= 0 || split_k < 0)
        return LOWM_ERR_INVALID_ARGUMENT;
    if (split_k != 0 && split_k != 1 && split_k != 2 && split_k != 3 && split_k != 4 && split_k != 8)
        return LOWM_ERR_INVALID_ARGUMENT;
    if (split_k == 0)
        split_k = choose_split_k(M, N, K, sms > 0 ? sms : 152);
    if (split_k == 0 || !shape_ok(M, N, K, split_k))
        return LOWM_ERR_UNSUPPORTED_SHAPE;
    const int kbt = K / lowm::kBlockK;                  // K blocks in all
    if (stages_override == 1)
        return LOWM_ERR_INVALID_ARGUMENT;
    const int nsm = sms > 0 ? sms : 152;
    const bool w_promise = (flags & LOWM_FLAG_W_BEFORE_PDL_WAIT) != 0;
    int tile_n = choose_tile_n(M, N, K, split_k, nsm);
    int m_pad = m_pad_for(M, tile_n);
    // The persistent schedule is opt-in (LOWM_PERSISTENT=1); it splits K evenly.
    bool persistent = env_int("LOWM_PERSISTENT", 0) == 1 && m_pad <= 64 && m_pad != 48 &&   // no persistent m_pad 48 / 96 / 128 instance
                      kbt % split_k == 0 && split_k != 3;
    int tiles = (N + tile_n - 1) / tile_n;            // the last tile may be partial
    int clusters = tiles;
    bool alias = false;
    Ring ring;
    int fp = 0;
    // The ring (and the mailbox placement) for one tile width: with the
    // mailbox in the ring when that is fixed, else whichever placement fits
    // the larger W ring (the separate mailbox on a tie: no hand-off needed).
    auto pick = [&]() {
        // Deep rings (and the mailbox in the ring, where that deepens it) with
        // the W promise or a stream of more than 512 KiB of W per CTA.  Short
        // streams without the promise keep the mailbox next to the ring unless
        // it must share it (M64 N6144 K4096 with default flags, before the
        // reduce-scatter mailbox: 2 x 3 next to the mailbox 12.17 us against
        // 4 x 2 in the ring 12.36 us); long ones gain from it (M16 N6144 K32768
        // split_k 4 on 128 columns: 2 x 3 in the ring, two CTAs per SM, 61.6
        // us against 2 x 2 next to the mailbox 63.8 us).
        const double per_cta_w = 2.0 * N * (double)K / ((double)tiles * split_k);
        const bool deep = w_promise || per_cta_w > kShortStreamBytes;
        int fa = forced_alias(m_pad, split_k);
        if (fa < 0 && !deep)
            fa = 0;
        auto one = [&](bool al, Ring &r, int &f) {
            r = choose_ring(tile_n, m_pad, split_k, kbt, tiles * split_k, nsm, 1, al, deep);
            if (stages_override >= 2)
                r.stages = stages_override;
            f = footprint(tile_n, m_pad, split_k, r.stages, r.kbs, 1, al);
        };
        if (fa >= 0) {
            alias = fa == 1;
            one(alias, ring, fp);
            return;
        }
        Ring r0, r1;
        int f0 = 0, f1 = 0;
        one(false, r0, f0);
        one(true, r1, f1);
        const long long w0 = f0 <= kMaxSmemPerCta ? (long long)r0.kbs * r0.stages : -1;
        const long long w1 = f1 <= kMaxSmemPerCta ? (long long)r1.kbs * r1.stages : -1;
        alias = w1 > w0;
        ring = alias ? r1 : r0;
        fp = alias ? f1 : f0;
    };
    pick();
    if (tile_n == 128 && (fp > kMaxSmemPerCta || !kernel_for(tile_n, m_pad, split_k, false))) {
        // e.g. m_pad 64 with split_k 8: the 128-column mailbox does not fit, or
        // m_pad 96 / 128 with split_k 4: no 128-column instance; use 64 columns
        tile_n = 64;
        m_pad = m_pad_of(M);
        tiles = (N + tile_n - 1) / tile_n;
        clusters = tiles;
        pick();
    }
    if (fp > kMaxSmemPerCta || !kernel_for(tile_n, m_pad, split_k, false))
        return LOWM_ERR_UNSUPPORTED_SHAPE;
    int smem = full_smem ? kMaxSmemPerCta : fp;
    if (persistent) {
        // Size the persistent grid for the CTAs that fit at the chosen footprint.
        Ring pr = choose_ring(tile_n, m_pad, split_k, kbt, tiles * split_k, nsm, 2);
        if (stages_override >= 2)
            pr.stages = stages_override;
        const int fp2 = footprint(tile_n, m_pad, split_k, pr.stages, pr.kbs, 2);
        if (fp2 <= kMaxSmemPerCta) {
            alias = false;
            ring = pr;
            fp = fp2;
            smem = full_smem ? kMaxSmemPerCta : fp;
            int fit = std::max(1, resident_clusters(tile_n, m_pad, split_k, smem, nsm, true, have_device));
            const int cap = env_int("LOWM_MAX_CLUSTERS", 0);   // tuning / test hook: fewer clusters
            if (cap > 0)
                fit = std::min(fit, cap);
            const int per = (tiles + std::min(tiles, fit) - 1) / std::min(tiles, fit);
            clusters = (tiles + per - 1) / per;          // every cluster gets `per` tiles (the last maybe fewer)
        } else {
            persistent = false;
        }
    }
    const int stages = ring.stages;
    const int kbs = ring.kbs;
    t->tile_n = tile_n;
    t->m_pad = m_pad;
    t->split_k = split_k;
    t->stages = stages;
    t->block_k = lowm::kBlockK;
    t->tiles = tiles;
    t->num_clusters = clusters;
    t->ctas = clusters * split_k;
    t->smem_bytes = smem;
    t->pdl = 1;
    t->persistent = persistent ? 1 : 0;
    t->tiles_per_cluster = (tiles + clusters - 1) / clusters;
    t->kb_per_stage = kbs;
    t->mma_issuers = persistent ? 1 : 2;
    t->mbox_in_ring = alias ? 1 : 0;
    // W stages requested ahead of the programmatic-dependency wait when the
    // caller promises that the preceding kernel does not write W: the whole
    // ring, except for rings of three or more 64-column stages on a grid
    // that overflows the SMs, where one stage measured fastest on GB300 (64
    // columns at M4 N6144 K4096, 192 CTAs: 9.95 us against 10.51 us for the
    // whole ring; the ring's next-GEMM requests otherwise slow the running
    // GEMM's tail).  With one CTA per SM the whole ring is best (M4 N6144 K4096
    // on a 4 x 3 128-column ring: 8.90 us against 9.81 with two stages and
    // 10.74 with one; M4 N2304 K12288 on an 8 x 3 ring: 9.98 against 10.73
    // with one).  LOWM_W_PREFETCH overrides (tuning).
    int wpf = (!persistent && tile_n == 64 && stages >= 3 && clusters * split_k > nsm) ? 1 : stages;
    const int force_wpf = env_int("LOWM_W_PREFETCH", -1);
    if (force_wpf >= 0)
        wpf = std::min(force_wpf, stages);
    t->w_prefetch_stages = w_promise ? wpf : 0;      // nothing is requested before the wait without the flag
    // W stages requested into L2 ahead of the newest ring load: one measured
    // fastest for every workload (GB300, interleaved repeats: M4 N6144 K4096
    // split_k 2 10.49 -> 10.15 us, M4 N2304 K12288 split_k 4 10.73 -> 9.95,
    // M64 11.37 -> 10.93, M128 14.51 -> 14.05, M4 N49152 60.78 -> 59.95);
    // two or more were slower than one almost everywhere.  LOWM_L2_PREFETCH
    // overrides (tuning).
    int l2pf = persistent ? 0 : 1;
    const int force_l2pf = env_int("LOWM_L2_PREFETCH", -1);
    if (force_l2pf >= 0 && !persistent)
        l2pf = force_l2pf;
    t->l2_prefetch_stages = l2pf;
    // Without the W promise nothing may land in shared memory before the
    // dependency wait, but W may be requested into L2 (every SM's stores
    // land there, so the line a later ring load reads is the current one):
    // one stage for a short stream, the whole ring for more than 512 KiB of
    // W per CTA (GB300, default flags, 0 -> 1 stage: M4 N6144 K4096 10.60 ->
    // 10.25 us, M64 11.37 -> 11.03; 0 -> 3: M4 N2304 K12288 split_k 4 11.69 ->
    // 11.25, M16 N6144 K32768 split_k 4 63.41 -> 62.76; two or more stages
    // lost on the short streams: 10.71 us at two).  LOWM_L2_BEFORE_WAIT
    // overrides (tuning).
    const double w_per_cta = 2.0 * N * (double)K / ((double)t->ctas);
    int l2bw = (w_promise || persistent) ? 0 : (w_per_cta > kShortStreamBytes ? t->stages : 1);
    const int force_l2bw = env_int("LOWM_L2_BEFORE_WAIT", -1);
    if (force_l2bw >= 0 && !w_promise && !persistent)
        l2bw = force_l2bw;
    t->l2_before_wait_stages = l2bw;
    return LOWM_OK;
}

// ------------------------------------------------------------------ TMA descriptors
struct MapKey {
    uintptr_t ptr;
    int rows, K, box_rows, box_kb;
    bool operator==(const MapKey &o) const
    {
        return ptr == o.ptr && rows == o.rows && K == o.K && box_rows == o.box_rows && box_kb == o.box_kb;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        size_t h = std::hash<uintptr_t>()(k.ptr);
        h ^= std::hash<long long>()(((long long)k.rows << 32) ^ ((long long)k.K << 12) ^ (k.box_rows << 4) ^
                                    k.box_kb) +
             0x9e3779b9 + (h << 6) + (h >> 2);
        return h;
    }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;   // guarded by g_mu

// 3-D view (k_inner, row, k_block) of a row-major [rows, K] bf16 matrix:
// extents {64, rows, K / 64}, byte strides {2K (row), 128 (k block)}.  A box
// {64, box_rows, box_kb} lands in shared memory as box_kb consecutive
// [box_rows x 64] tiles with 128-byte swizzling, the layout the MMA
// descriptors expect.  Rows beyond `rows` are zero-filled.
lowm_status_t get_map(const void *ptr, int rows, int K, int box_rows, int box_kb, CUtensorMap *out)
{
    const MapKey key{reinterpret_cast<uintptr_t>(ptr), rows, K, box_rows, box_kb};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return LOWM_OK;
        }
    }
    EncodeTiledFn enc = get_encode_fn();
    if (!enc)
        return LOWM_ERR_CUDA;
    CUtensorMap m;
    std::memset(&m, 0, sizeof m);
    const cuuint64_t dims[3] = {(cuuint64_t)lowm::kBlockK, (cuuint64_t)rows, (cuuint64_t)(K / lowm::kBlockK)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)lowm::kBlockK * 2};
    const cuuint32_t box[3] = {(cuuint32_t)lowm::kBlockK, (cuuint32_t)box_rows, (cuuint32_t)box_kb};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return LOWM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_maps.size() > 4096)
        g_maps.clear();
    g_maps.emplace(key, m);
    *out = m;
    return LOWM_OK;
}

// ------------------------------------------------------------------ launch
bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

lowm_status_t launch(const void *A, const void *W, void *C, int M, int N, int K, int split_k, void *stream,
                     const lowm_debug_opts_t *dbg, unsigned int flags = 0)
{
    if (flags & ~(LOWM_FLAG_W_BEFORE_PDL_WAIT | LOWM_FLAG_A_BEFORE_PDL_WAIT))
        return LOWM_ERR_INVALID_ARGUMENT;
    if (!A || !W || !C)
        return LOWM_ERR_INVALID_ARGUMENT;
    if (M <= 0 || N <= 0 || K <= 0)
        return LOWM_ERR_INVALID_ARGUMENT;
    if (!aligned16(A) || !aligned16(W) || !aligned16(C))
        return LOWM_ERR_MISALIGNED;
    const size_t a_bytes = (size_t)M * K * 2, w_bytes = (size_t)N * K * 2, c_bytes = (size_t)M * N * 2;
    if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, W, w_bytes))
        return LOWM_ERR_INVALID_ARGUMENT;
    if (dbg && (dbg->stages == 1 || dbg->stages < 0))
        return LOWM_ERR_INVALID_ARGUMENT;
    int sms = 0;
    lowm_status_t st = check_device(&sms);
    if (st != LOWM_OK)
        return st;
    lowm_tactic_t t;
    st = make_tactic(M, N, K, split_k, sms, true, flags, dbg ? dbg->stages : 0, (dbg && dbg->full_smem) ? 1 : 0, &t);
    if (st != LOWM_OK)
        return st;
    KernelFn fn = kernel_for(t.tile_n, t.m_pad, t.split_k, t.persistent != 0);
    if (!fn)
        return LOWM_ERR_UNSUPPORTED_SHAPE;
    if ((st = prepare_kernel(fn)) != LOWM_OK)
        return st;
    CUtensorMap map_a, map_w;
    if ((st = get_map(A, M, K, t.m_pad, t.kb_per_stage, &map_a)) != LOWM_OK)
        return st;
    if ((st = get_map(W, N, K, t.tile_n, t.kb_per_stage, &map_w)) != LOWM_OK)
        return st;

    KernelParams p;
    std::memset(&p, 0, sizeof p);
    p.C = reinterpret_cast<__nv_bfloat16 *>(C);
    p.status = status_word();
    if (!p.status)
        return LOWM_ERR_CUDA;
    p.M = M;
    p.N = N;
    p.K = K;
    p.stages = t.stages;
    p.kb_per_rank = K / (t.split_k * lowm::kBlockK);
    p.kb_per_stage = t.kb_per_stage;
    p.stages_total = K / (lowm::kBlockK * t.kb_per_stage);
    p.mbox_in_ring = t.mbox_in_ring ? 1u : 0u;
    p.num_tiles = t.tiles;
    p.timeout_ns = lowm::kDefaultTimeoutNs;
    p.reduce_timeout_ns = lowm::kDefaultTimeoutNs;
    p.w_prefetch_stages = (uint32_t)t.w_prefetch_stages;   // 0 unless the flag is set
    p.l2_prefetch_stages = (uint32_t)t.l2_prefetch_stages;
    p.l2_before_wait_stages = (uint32_t)t.l2_before_wait_stages;
    // Loads skip the dependency wait only when neither operand is written by
    // the preceding kernel (both promises); C still waits in the epilogue.
    constexpr unsigned kBoth = LOWM_FLAG_W_BEFORE_PDL_WAIT | LOWM_FLAG_A_BEFORE_PDL_WAIT;
    p.a_before_wait = (flags & kBoth) == kBoth ? 1u : 0u;
    if (dbg) {
        p.stall_warp_mask = dbg->stall_warp_mask;
        p.stall_rank_mask = dbg->stall_rank_mask;
        p.stall_ns = dbg->stall_ns;
        p.drop_mailbox = dbg->drop_mailbox ? 1u : 0u;
        p.probes = dbg->probes;
        p.c_f32 = dbg->c_f32;
        p.timeline = dbg->timeline;
        if (dbg->reduce_timeout_ns)
            p.reduce_timeout_ns = dbg->reduce_timeout_ns;
    }

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)t.ctas, 1, 1);
    cfg.blockDim = dim3((unsigned)(t.persistent ? lowm::kThreadsPersistent : lowm::kThreads), 1, 1);
    cfg.dynamicSmemBytes = (size_t)t.smem_bytes;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attrs[3];
    int na = 0;
    if (t.split_k > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)t.split_k;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
        // Tuning hook: LOWM_CLUSTER_POLICY = 1 (spread) or 2 (load balancing).
        const int pol = env_int("LOWM_CLUSTER_POLICY", 0);
        if (pol == 1 || pol == 2) {
            attrs[na].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
            attrs[na].val.clusterSchedulingPolicyPreference =
                pol == 1 ? cudaClusterSchedulingPolicySpread : cudaClusterSchedulingPolicyLoadBalancing;
            ++na;
        }
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = (unsigned)na;
    if (std::getenv("LOWM_LOG"))
        std::fprintf(stderr,
                     "lowm: M%d N%d K%d -> tile_n %d m_pad %d split_k %d stages %d x %d blocks ctas %d smem %d "
                     "persistent %d mbox_in_ring %d\n",
                     M, N, K, t.tile_n, t.m_pad, t.split_k, t.stages, t.kb_per_stage, t.ctas, t.smem_bytes,
                     t.persistent, t.mbox_in_ring);
    if (cudaLaunchKernelEx(&cfg, fn, map_a, map_w, p) != cudaSuccess)
        return LOWM_ERR_CUDA;
    return LOWM_OK;
}

}  // namespace

extern "C" {

lowm_status_t lowm_gemm_bf16(const void *A, const void *W, void *C, int M, int N, int K, int split_k, void *stream)
{
    return launch(A, W, C, M, N, K, split_k, stream, nullptr);
}

lowm_status_t lowm_gemm_bf16_ex(const void *A, const void *W, void *C, int M, int N, int K, int split_k,
                                unsigned int flags, void *stream)
{
    return launch(A, W, C, M, N, K, split_k, stream, nullptr, flags);
}

lowm_status_t lowm_gemm_bf16_debug(const void *A, const void *W, void *C, int M, int N, int K, int split_k,
                                   void *stream, const lowm_debug_opts_t *opts)
{
    return launch(A, W, C, M, N, K, split_k, stream, opts, opts ? opts->flags : 0u);
}

lowm_status_t lowm_gemm_query_tactic(int M, int N, int K, int split_k, lowm_tactic_t *out)
{
    return lowm_gemm_query_tactic_ex(M, N, K, split_k, 0u, out);
}

lowm_status_t lowm_gemm_query_tactic_ex(int M, int N, int K, int split_k, unsigned int flags, lowm_tactic_t *out)
{
    if (!out)
        return LOWM_ERR_INVALID_ARGUMENT;
    if (flags & ~(LOWM_FLAG_W_BEFORE_PDL_WAIT | LOWM_FLAG_A_BEFORE_PDL_WAIT))
        return LOWM_ERR_INVALID_ARGUMENT;
    // Host-only query: with a usable sm_103 device current, the same numbers the
    // launch uses; otherwise the per-SM arithmetic for a 152-SM GB300.
    int sms = 152;
    int n = 0;
    bool have_device = false;
    if (cudaGetDeviceCount(&n) == cudaSuccess && n > 0)
        have_device = check_device(&sms) == LOWM_OK;
    if (!have_device) {
        cudaGetLastError();
        sms = 152;
    }
    lowm_tactic_t t;
    const lowm_status_t st = make_tactic(M, N, K, split_k, sms, have_device, flags, 0, 0, &t);
    if (st == LOWM_OK)
        *out = t;
    return st;
}

const char *lowm_status_string(lowm_status_t s)
{
    switch (s) {
    case LOWM_OK: return "ok";
    case LOWM_ERR_INVALID_ARGUMENT: return "invalid argument";
    case LOWM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (need 1<=M<=128, N>=1, K a multiple of 64 with K/64>=split_k, and a split-K mailbox that fits)";
    case LOWM_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case LOWM_ERR_UNSUPPORTED_ARCH: return "current device is not sm_103 (GB300)";
    case LOWM_ERR_CUDA: return "CUDA runtime error";
    case LOWM_ERR_TIMEOUT: return "a kernel wait timed out";
    }
    return "unknown status";
}

lowm_status_t lowm_gemm_sync_status(void *stream, unsigned int *detail)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LOWM_ERR_CUDA;
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, lowm::g_lowm_status, sizeof v) != cudaSuccess)
        return LOWM_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(lowm::g_lowm_status, &zero, sizeof zero) != cudaSuccess)
        return LOWM_ERR_CUDA;
    if (detail)
        *detail = v;
    return v ? LOWM_ERR_TIMEOUT : LOWM_OK;
}

lowm_status_t lowm_gemm_bf16_host(const void *A_host, const void *W_host, void *C_host, void *A_dev, void *W_dev,
                                  void *C_dev, int M, int N, int K, int split_k, void *stream)
{
    if (!A_host || !W_host || !C_host || !A_dev || !W_dev || !C_dev)
        return LOWM_ERR_INVALID_ARGUMENT;
    if (M <= 0 || N <= 0 || K <= 0)
        return LOWM_ERR_INVALID_ARGUMENT;
    lowm_tactic_t t;
    int sms = 0;
    lowm_status_t st = check_device(&sms);
    if (st != LOWM_OK)
        return st;
    if ((st = make_tactic(M, N, K, split_k, sms, true, 0u, 0, 0, &t)) != LOWM_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(A_dev, A_host, (size_t)M * K * 2, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(W_dev, W_host, (size_t)N * K * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return LOWM_ERR_CUDA;
    if ((st = launch(A_dev, W_dev, C_dev, M, N, K, split_k, stream, nullptr)) != LOWM_OK)
        return st;
    if (cudaMemcpyAsync(C_host, C_dev, (size_t)M * N * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return LOWM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return LOWM_ERR_CUDA;
    return LOWM_OK;
}

lowm_status_t lowm_tmem_hog_launch(void *stream, int ctas, int ncols, int iters)
{
    if (ctas <= 0 || iters < 0 || ncols < 32 || ncols > 256 || (ncols & (ncols - 1)) != 0)
        return LOWM_ERR_INVALID_ARGUMENT;
    lowm_status_t st = check_device(nullptr);
    if (st != LOWM_OK)
        return st;
    lowm::tmem_hog_kernel<<<ctas, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ncols, iters);
    return cudaGetLastError() == cudaSuccess ? LOWM_OK : LOWM_ERR_CUDA;
}

}  // extern "C"
