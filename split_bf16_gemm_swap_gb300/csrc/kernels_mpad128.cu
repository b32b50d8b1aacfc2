// Kernel instances for m_pad 128 (65 <= M <= 128), one-tile-per-cluster
// schedule only.  The split-K mailbox holds (split_k - 1) x tile_n x 128 fp32:
// next to the ring, 64-column tiles fit up to split_k 4 and 128-column tiles
// up to split_k 2 in one CTA's shared memory; split_k 3 places the mailbox in
// the drained ring.
#include "lowm_kernels.h"

namespace lowm {

KernelFn kernel_mpad128(int tile_n, int split_k)
{
    if (tile_n == 64) {
        switch (split_k) {
        case 1: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 128, 1>);
        case 2: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 128, 2>);
        case 3: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 128, 3>);
        case 4: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 128, 4>);
        default: return nullptr;
        }
    }
    if (tile_n == 128) {
        switch (split_k) {
        case 1: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<128, 128, 1>);
        case 2: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<128, 128, 2>);
        case 3: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<128, 128, 3>);
        default: return nullptr;
        }
    }
    return nullptr;
}

}  // namespace lowm
