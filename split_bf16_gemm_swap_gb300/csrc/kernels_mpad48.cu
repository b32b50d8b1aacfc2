// Kernel instances for m_pad 48 (33 <= M <= 48), one-tile-per-cluster
// schedule only: the MMA's N is 48 (a multiple of 16, so both tile widths),
// a quarter fewer activation bytes per stage and per mailbox slot than m_pad
// 64.  split_k 2 with the mailbox next to the ring exchanges as a
// reduce-scatter of two 24-row halves.
#include "lowm_kernels.h"

namespace lowm {
namespace {

template <int TN>
KernelFn by_split48(int split_k)
{
    switch (split_k) {
    case 1: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<TN, 48, 1>);
    case 2: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<TN, 48, 2>);
    case 3: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<TN, 48, 3>);
    case 4: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<TN, 48, 4>);
    case 8: return reinterpret_cast<KernelFn>(&lowm_splitk_kernel<TN, 48, 8>);
    default: return nullptr;
    }
}

}  // namespace

KernelFn kernel_mpad48(int tile_n, int split_k)
{
    if (tile_n == 64)
        return by_split48<64>(split_k);
    if (tile_n == 128)
        return by_split48<128>(split_k);
    return nullptr;
}

}  // namespace lowm
