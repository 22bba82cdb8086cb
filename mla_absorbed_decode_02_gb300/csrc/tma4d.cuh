// 4-D tiled TMA load (the projection and extend kernels read weights and workspaces through
// 4-D views so that one copy brings several 64-column blocks).
#pragma once
#include "common.cuh"

namespace mla {

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            int w, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
      : "memory");
}

}  // namespace mla
