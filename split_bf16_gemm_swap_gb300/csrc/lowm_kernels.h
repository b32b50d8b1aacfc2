// Internal interface between the host launcher and the kernel instances,
// which are compiled in separate translation units (one per tile width) so
// the library builds in parallel.
#pragma once

#include <cuda.h>

#include "lowm_kernel.cuh"

namespace lowm {

typedef void (*KernelFn)(CUtensorMap, CUtensorMap, KernelParams);

// The kernel for (m_pad, split_k, persistent) at 64-column tiles (m_pad 8, 16,
// 32, 64) and at 128-column tiles (m_pad 16, 32, 64); split_k 3 has no
// persistent instance; nullptr when no instance exists.
KernelFn kernel_tile64(int m_pad, int split_k, bool persistent);
KernelFn kernel_tile128(int m_pad, int split_k, bool persistent);
// m_pad 128 (one-tile schedule): tile_n 64 with split_k 1, 2, 3, 4; tile_n 128
// with split_k 1, 2, 3; nullptr otherwise.
KernelFn kernel_mpad128(int tile_n, int split_k);
// m_pad 96 (65 <= M <= 96), the same instances as m_pad 128.
KernelFn kernel_mpad96(int tile_n, int split_k);
// m_pad 48 (33 <= M <= 48), one-tile schedule, split_k 1, 2, 3, 4, 8 at both
// tile widths.
KernelFn kernel_mpad48(int tile_n, int split_k);

}  // namespace lowm
