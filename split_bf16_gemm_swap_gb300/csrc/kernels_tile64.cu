// Kernel instances for 64-column tiles (MMA M = 64).
#include "lowm_kernels.h"
#include "lowm_persistent.cuh"

namespace lowm {
namespace {

template <int MP, int SK>
KernelFn instance(bool persistent)
{
    return persistent ? reinterpret_cast<KernelFn>(&lowm_splitk_persistent_kernel<64, MP, SK>)
                      : reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, MP, SK>);
}

template <int MP>
KernelFn by_split(int split_k, bool persistent)
{
    switch (split_k) {
    case 1: return instance<MP, 1>(persistent);
    case 2: return instance<MP, 2>(persistent);
    case 3:   // uneven K split; one-tile schedule only
        return persistent ? nullptr : reinterpret_cast<KernelFn>(&lowm_splitk_kernel<64, MP, 3>);
    case 4: return instance<MP, 4>(persistent);
    case 8: return instance<MP, 8>(persistent);
    default: return nullptr;
    }
}

}  // namespace

KernelFn kernel_tile64(int m_pad, int split_k, bool persistent)
{
    switch (m_pad) {
    case 8: return by_split<8>(split_k, persistent);
    case 16: return by_split<16>(split_k, persistent);
    case 32: return by_split<32>(split_k, persistent);
    case 64: return by_split<64>(split_k, persistent);
    default: return nullptr;
    }
}

}  // namespace lowm
