// Kernel instances for m_pad 96 (65 <= M <= 96), one-tile-per-cluster
// schedule only: the MMA's N is 96 (a multiple of 16, so both tile widths),
// a quarter fewer activation bytes per stage and per mailbox slot than m_pad
// 128, and the same chunked epilogue with three 32-column chunks.
#include "lowm_kernels.h"

namespace lowm {

KernelFn kernel_mpad96(int tile_n, int split_k)
{
    if (tile_n == 64) {
        switch (split_k) {
        case 1: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 96, 1>);
        case 2: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 96, 2>);
        case 3: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 96, 3>);
        case 4: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, 96, 4>);
        default: return nullptr;
        }
    }
    if (tile_n == 128) {
        switch (split_k) {
        case 1: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<128, 96, 1>);
        case 2: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<128, 96, 2>);
        case 3: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<128, 96, 3>);
        default: return nullptr;
        }
    }
    return nullptr;
}

}  // namespace lowm
